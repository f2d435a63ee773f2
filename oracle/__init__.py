"""CPU oracle for the UltraQuant 4-bit KV cache (test infrastructure).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline and
reference legs may import this package.  The product library never calls it and
shares no code with it; see uq_oracle.c for the step-by-step restatement of the
pages and the readings taken where they are silent.

All arrays are numpy.  bf16 tensors are passed as uint16 bit patterns.
"""
import ctypes as C

import numpy as np

from .build import build as _build

_lib = C.CDLL(_build())

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_i8p = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")

_lib.uqo_splitmix64.restype = C.c_uint64
_lib.uqo_splitmix64.argtypes = [C.c_uint64, C.c_uint64]
_lib.uqo_signs.argtypes = [C.c_uint64, C.c_int, _i8p]
_lib.uqo_inv_sqrt_d.restype = C.c_float
_lib.uqo_inv_sqrt_d.argtypes = [C.c_int]
_lib.uqo_rotate_fp32.argtypes = [_f32p, C.c_int, _i8p, _f32p]
_lib.uqo_inverse_rotate_f64.argtypes = [_f64p, C.c_int, _i8p, _f64p]
_lib.uqo_inverse_rotate_fp32.argtypes = [_f32p, C.c_int, _i8p, _f32p]
_lib.uqo_pow2_exponent.restype = C.c_int
_lib.uqo_pow2_exponent.argtypes = [C.c_double, C.c_int]
_lib.uqo_scale_byte.restype = C.c_int
_lib.uqo_scale_byte.argtypes = [C.c_float, C.c_float, C.c_int]
_lib.uqo_e2m1_code.restype = C.c_int
_lib.uqo_e2m1_code.argtypes = [C.c_double]
_lib.uqo_e2m1_value.restype = C.c_double
_lib.uqo_e2m1_value.argtypes = [C.c_int]
_lib.uqo_fp4_value.restype = C.c_double
_lib.uqo_fp4_value.argtypes = [C.c_int, C.c_int]
_lib.uqo_quantize_rotated.argtypes = [_f32p, C.c_int64, C.c_int, C.c_float, C.c_int, _u8p, _u8p]
_lib.uqo_c_constant.restype = C.c_float
_lib.uqo_quantize_vectors.argtypes = [C.c_void_p, C.c_int, C.c_int64, C.c_int, C.c_uint64, _u8p, _u8p]
_lib.uqo_f32_to_bf16.restype = C.c_uint16
_lib.uqo_f32_to_bf16.argtypes = [C.c_float]
_lib.uqo_e4m3_value.restype = C.c_double
_lib.uqo_e4m3_value.argtypes = [C.c_int]
_lib.uqo_e4m3_code.restype = C.c_int
_lib.uqo_e4m3_code.argtypes = [C.c_float]
_lib.uqo_query_fp8.argtypes = [_u16p, C.c_int, C.c_uint64, _u8p]
_lib.uqo_append_fp4.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int64, _i64p, C.c_int, C.c_int,
                                C.c_int, C.c_uint64, _u8p, _u8p, _u8p, _u8p]
_lib.uqo_append_fp4_c.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int64, _i64p, C.c_int, C.c_int,
                                  C.c_int, C.c_uint64, C.c_float, _u8p, _u8p, _u8p, _u8p]
_lib.uqo_append_fp8.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int64, _i64p, C.c_int, C.c_int,
                                C.c_int, C.c_float, C.c_float, _u8p, _u8p]
_lib.uqo_append_bf16.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int64, _i64p, C.c_int, C.c_int,
                                 C.c_int, _u16p, _u16p]
_lib.uqo_decode.argtypes = [C.c_int, _u16p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_float, C.c_float,
                            _i32p, C.c_int, _i32p, C.c_double, C.c_uint64, _f64p]

_lib.uqo_decode_ex.argtypes = [C.c_int, _u16p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_float, C.c_float,
                               _i32p, C.c_int, _i32p, C.c_double, C.c_uint64, C.c_void_p, _f64p]
_lib.uqo_f16_round.restype = C.c_double
_lib.uqo_f16_round.argtypes = [C.c_float]
_lib.uqo_tq_norm.restype = C.c_double
_lib.uqo_tq_norm.argtypes = [_f32p, C.c_int]
_lib.uqo_tq_code.restype = C.c_int
_lib.uqo_tq_code.argtypes = [C.c_double, _f64p]
_lib.uqo_tq_value.restype = C.c_double
_lib.uqo_tq_value.argtypes = [C.c_int, _f64p]
_lib.uqo_tq_quantize_row.argtypes = [_f32p, C.c_int, _i8p, _f64p, _u8p, _f32p]
_lib.uqo_append_tq4.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int64, _i64p, C.c_int, C.c_int,
                                C.c_int, C.c_uint64, _f64p, _u8p, _f32p, _u8p, _f32p]
_lib.uqo_query_f16.argtypes = [_u16p, C.c_int, C.c_uint64, _f64p]

KIND_FP4, KIND_FP8, KIND_BF16, KIND_TQ4 = 0, 1, 2, 3
DEFAULT_SEED = 42
C_CONSTANT = float(_lib.uqo_c_constant())
ROUND_LOG2, ROUND_LINEAR, ROUND_FLOOR, ROUND_CEIL = 0, 1, 2, 3


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def splitmix64(seed: int, i: int) -> int:
    return int(_lib.uqo_splitmix64(seed, i))


def signs(seed: int, d: int) -> np.ndarray:
    s = np.empty(d, np.int8)
    _lib.uqo_signs(seed, d, s)
    return s


def inv_sqrt_d(d: int) -> np.float32:
    return np.float32(_lib.uqo_inv_sqrt_d(d))


def rotate_fp32(x: np.ndarray, seed: int = DEFAULT_SEED) -> np.ndarray:
    """R1 forward rotation of each row of x (fp32)."""
    x = _c(x, np.float32)
    d = x.shape[-1]
    s = signs(seed, d)
    flat = x.reshape(-1, d)
    out = np.empty_like(flat)
    for r in range(flat.shape[0]):
        _lib.uqo_rotate_fp32(flat[r], d, s, out[r])
    return out.reshape(x.shape)


def inverse_rotate_f64(o: np.ndarray, seed: int = DEFAULT_SEED) -> np.ndarray:
    o = _c(o, np.float64)
    d = o.shape[-1]
    s = signs(seed, d)
    flat = o.reshape(-1, d)
    out = np.empty_like(flat)
    for r in range(flat.shape[0]):
        _lib.uqo_inverse_rotate_f64(flat[r], d, s, out[r])
    return out.reshape(o.shape)


def inverse_rotate_fp32(o: np.ndarray, seed: int = DEFAULT_SEED) -> np.ndarray:
    """fp32 inverse rotation s .* fl32(FWHT_fp32(o) * fl32(1/sqrt d)) of each row
    (the decode's output stage)."""
    o = _c(o, np.float32)
    d = o.shape[-1]
    s = signs(seed, d)
    flat = o.reshape(-1, d)
    out = np.empty_like(flat)
    for r in range(flat.shape[0]):
        _lib.uqo_inverse_rotate_fp32(flat[r], d, s, out[r])
    return out.reshape(o.shape)


def pow2_exponent(t: float, mode: int = ROUND_LOG2) -> int:
    return int(_lib.uqo_pow2_exponent(float(t), mode))


def scale_byte(m: float, c: float = None, mode: int = ROUND_LOG2) -> int:
    return int(_lib.uqo_scale_byte(np.float32(m), np.float32(C_CONSTANT if c is None else c), mode))


def e2m1_code(r: float) -> int:
    return int(_lib.uqo_e2m1_code(float(r)))


def e2m1_value(code: int) -> float:
    return float(_lib.uqo_e2m1_value(code))


def fp4_value(code: int, byte: int) -> float:
    return float(_lib.uqo_fp4_value(code, byte))


def quantize_rotated(y: np.ndarray, c: float = None, mode: int = ROUND_LOG2):
    """Quantiser stage alone (R2 + R3) on already-rotated rows."""
    y = _c(y, np.float32)
    d = y.shape[-1]
    n = y.size // d
    codes = np.empty(n * d // 2, np.uint8)
    scales = np.empty(n * d // 32, np.uint8)
    _lib.uqo_quantize_rotated(y.reshape(-1), n, d, np.float32(C_CONSTANT if c is None else c), mode,
                              codes, scales)
    return codes.reshape(y.shape[:-1] + (d // 2,)), scales.reshape(y.shape[:-1] + (d // 32,))


def _rows(x):
    """(pointer-holding array, is_fp32) for a bf16 (uint16) or fp32 array."""
    if x.dtype == np.uint16:
        return _c(x, np.uint16), 0
    return _c(x, np.float32), 1


def quantize_vectors(x: np.ndarray, seed: int = DEFAULT_SEED):
    """R1 + R2 + R3 on rows of x (uint16 bf16 bits or fp32)."""
    xa, f32 = _rows(x)
    d = xa.shape[-1]
    n = xa.size // d
    codes = np.empty(n * d // 2, np.uint8)
    scales = np.empty(n * d // 32, np.uint8)
    _lib.uqo_quantize_vectors(xa.ctypes.data, f32, n, d, seed, codes, scales)
    return codes.reshape(xa.shape[:-1] + (d // 2,)), scales.reshape(xa.shape[:-1] + (d // 32,))


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32).reshape(-1)
    return np.array([_lib.uqo_f32_to_bf16(v) for v in x], np.uint16)


def e4m3_value(byte: int) -> float:
    return float(_lib.uqo_e4m3_value(byte))


def e4m3_code(x: float) -> int:
    return int(_lib.uqo_e4m3_code(np.float32(x)))


def query_fp8(q_bf16: np.ndarray, seed: int = DEFAULT_SEED) -> np.ndarray:
    """R4: rotated E4M3 query bytes for each bf16 row."""
    q = _c(q_bf16, np.uint16)
    d = q.shape[-1]
    flat = q.reshape(-1, d)
    out = np.empty(flat.shape, np.uint8)
    for r in range(flat.shape[0]):
        _lib.uqo_query_fp8(flat[r], d, seed, out[r])
    return out.reshape(q.shape)


class Cache:
    """Host copy of a paged cache in the library's layout [P][Hkv][ps][row]."""

    def __init__(self, kind, num_pages, num_kv_heads, page_size, head_dim, k_scale=1.0, v_scale=1.0,
                 seed=DEFAULT_SEED, c=None):
        """c: the FP4 scale-rule constant (None: the pages' 0.156)."""
        self.kind, self.P, self.Hkv, self.ps, self.d = kind, num_pages, num_kv_heads, page_size, head_dim
        self.k_scale, self.v_scale, self.seed = float(k_scale), float(v_scale), seed
        self.c = C_CONSTANT if c is None else float(c)
        rows = num_pages * num_kv_heads * page_size
        if kind == KIND_FP4:
            self.kc = np.zeros((rows, head_dim // 2), np.uint8)
            self.vc = np.zeros((rows, head_dim // 2), np.uint8)
            self.ks = np.zeros((rows, head_dim // 32), np.uint8)
            self.vs = np.zeros((rows, head_dim // 32), np.uint8)
        elif kind == KIND_TQ4:
            self.kc = np.zeros((rows, head_dim // 2), np.uint8)
            self.vc = np.zeros((rows, head_dim // 2), np.uint8)
            self.ks = np.zeros(rows, np.float32)  # norms
            self.vs = np.zeros(rows, np.float32)
            self.cpos = tq_centroids(head_dim)   # fp64 centroids of the non-negative half
            self.mags = self.cpos                # the decode's reconstruction table (see decode)
        elif kind == KIND_FP8:
            self.kc = np.zeros((rows, head_dim), np.uint8)
            self.vc = np.zeros((rows, head_dim), np.uint8)
            self.ks = self.vs = None
        else:
            self.kc = np.zeros((rows, head_dim), np.uint16)
            self.vc = np.zeros((rows, head_dim), np.uint16)
            self.ks = self.vs = None

    def append(self, k, v, slot_mapping):
        """Quantize-append T tokens ([T][Hkv][d], bf16 bits or fp32)."""
        ka, f32 = _rows(k)
        va, _ = _rows(v)
        T = ka.shape[0]
        slots = _c(slot_mapping, np.int64)
        args = (ka.ctypes.data, va.ctypes.data, f32, T, slots, self.Hkv, self.ps, self.d)
        if self.kind == KIND_FP4:
            _lib.uqo_append_fp4_c(*args, self.seed, np.float32(self.c), self.kc, self.ks, self.vc, self.vs)
        elif self.kind == KIND_TQ4:
            _lib.uqo_append_tq4(*args, self.seed, _c(self.cpos, np.float64), self.kc, self.ks, self.vc, self.vs)
        elif self.kind == KIND_FP8:
            _lib.uqo_append_fp8(*args, np.float32(self.k_scale), np.float32(self.v_scale), self.kc, self.vc)
        else:
            _lib.uqo_append_bf16(*args, self.kc, self.vc)

    def decode(self, q_bf16, block_table, seq_lens, sm_scale=0.0, tq_table=None):
        """fp64 decode attention; q: [B][Hq][d] bf16 bits -> [B][Hq][d] float64.
        TQ4: values are code -> +-table[rank] x norm, the table being the fp64
        centroids unless tq_table (8 non-negative magnitudes) is given."""
        q = _c(q_bf16, np.uint16)
        B, Hq, d = q.shape
        bt = _c(block_table, np.int32)
        sl = _c(seq_lens, np.int32)
        out = np.empty((B, Hq, d), np.float64)
        ptr = lambda a: None if a is None else a.ctypes.data
        mags = None
        if self.kind == KIND_TQ4:
            mags = _c(self.mags if tq_table is None else tq_table, np.float64)
        _lib.uqo_decode_ex(self.kind, q.reshape(-1), B, Hq, self.Hkv, d, self.ps, ptr(self.kc), ptr(self.ks),
                           ptr(self.vc), ptr(self.vs), np.float32(self.k_scale), np.float32(self.v_scale),
                           bt.reshape(-1), bt.shape[1], sl, float(sm_scale), self.seed, ptr(mags),
                           out.reshape(-1))
        return out


_lib.uqo_e2m1_codes.argtypes = [_f64p, C.c_int64, _u8p]
_lib.uqo_e4m3_codes.argtypes = [_f32p, C.c_int64, _u8p]
_lib.uqo_scale_bytes.argtypes = [_f32p, C.c_int64, C.c_float, C.c_int, _u8p]
_lib.uqo_group_mse.restype = C.c_double
_lib.uqo_group_mse.argtypes = [_f32p, C.c_int64, C.c_float, C.c_int]
ROUND_CONTINUOUS = -1


_lib.uqo_e2m1_codes_bits.argtypes = [C.c_uint32, C.c_int64, _u8p]
_lib.uqo_scale_bytes_bits.argtypes = [C.c_uint32, C.c_int64, C.c_float, _u8p]


def e2m1_codes_of_bits(first: int, n: int) -> np.ndarray:
    """R3 code of the fp32 values with bit patterns first .. first + n - 1 (NaN: 0xFF)."""
    assert 0 <= first and first + n <= 1 << 32
    out = np.empty(n, np.uint8)
    _lib.uqo_e2m1_codes_bits(first, n, out)
    return out


def scale_bytes_of_bits(first: int, n: int, c: float = None) -> np.ndarray:
    """R2 byte of a group with absolute maximum |value| for the fp32 bit patterns first .. first + n - 1."""
    assert 0 <= first and first + n <= 1 << 32
    out = np.empty(n, np.uint8)
    _lib.uqo_scale_bytes_bits(first, n, np.float32(C_CONSTANT if c is None else c), out)
    return out


def e2m1_codes(r: np.ndarray) -> np.ndarray:
    r = _c(r, np.float64).reshape(-1)
    out = np.empty(r.size, np.uint8)
    _lib.uqo_e2m1_codes(r, r.size, out)
    return out


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32).reshape(-1)
    out = np.empty(x.size, np.uint8)
    _lib.uqo_e4m3_codes(x, x.size, out)
    return out


def scale_bytes(m: np.ndarray, c: float = None, mode: int = ROUND_LOG2) -> np.ndarray:
    m = _c(m, np.float32).reshape(-1)
    out = np.empty(m.size, np.uint8)
    _lib.uqo_scale_bytes(m, m.size, np.float32(C_CONSTANT if c is None else c), mode, out)
    return out


def group_mse(y: np.ndarray, c: float, mode: int) -> float:
    y = _c(y, np.float32).reshape(-1)
    return float(_lib.uqo_group_mse(y, y.size // 32, np.float32(c), mode))

_lib.uqo_kbyte_pos.restype = C.c_int
_lib.uqo_kbyte_pos.argtypes = [C.c_int, C.c_int]


def kbyte_pos(j: int, d: int) -> int:
    """Cache position of natural code byte j of a K row (group-interleaved words)."""
    return int(_lib.uqo_kbyte_pos(j, d))


# ---------------------------------------------------------------- TQ4 (TurboQuant codebook variant)
_TQ_BOOKS = {}


def tq_codebook(d: int, bits: int = 4):
    """(f16 magnitudes c_8..c_15 as float64, fp32 thresholds tau_0..tau_14):
    the f16 / fp32 roundings of the Lloyd-Max codebook for head_dim d
    (oracle/tq.py), the form in which the library stores its table; cached."""
    from . import tq
    key = (d, bits)
    if key not in _TQ_BOOKS:
        _TQ_BOOKS[key] = tq.codebook(d, bits)
    return _TQ_BOOKS[key]


def tq_centroids(d: int) -> np.ndarray:
    """fp64 centroids c_8 < ... < c_15 of the non-negative half of the 4-bit
    Lloyd-Max codebook (oracle/tq.py): the oracle's quantiser and default
    reconstruction table."""
    from . import tq
    key = (d, "c64")
    if key not in _TQ_BOOKS:
        _TQ_BOOKS[key] = np.ascontiguousarray(tq.lloyd_max(d, 4)[8:], np.float64)
    return _TQ_BOOKS[key]


def f16_round(x: float) -> float:
    return float(_lib.uqo_f16_round(np.float32(x)))


def tq_norm(y: np.ndarray) -> float:
    """fp64 Euclidean norm of a rotated row (T3)."""
    y = _c(y, np.float32)
    return float(_lib.uqo_tq_norm(y, y.size))


def tq_code(u: float, cpos: np.ndarray) -> int:
    """T4: sign-magnitude nibble of the centroid nearest to u."""
    return int(_lib.uqo_tq_code(float(u), _c(cpos, np.float64)))


def tq_value(code: int, mags: np.ndarray) -> float:
    return float(_lib.uqo_tq_value(code, _c(mags, np.float64)))


def tq_quantize_rows(x: np.ndarray, seed: int = DEFAULT_SEED):
    """Rotate + TQ4-quantise rows of x (fp32 or bf16 bits): (codes [n][d/2]
    natural byte order, norms [n] fp32)."""
    xa, f32 = _rows(x)
    d = xa.shape[-1]
    flat = xa.reshape(-1, d)
    if not f32:
        flat = (flat.astype(np.uint32) << 16).view(np.float32)
    flat = _c(flat, np.float32)
    cpos = tq_centroids(d)
    s = signs(seed, d)
    codes = np.empty((flat.shape[0], d // 2), np.uint8)
    norms = np.empty(flat.shape[0], np.float32)
    for r in range(flat.shape[0]):
        _lib.uqo_tq_quantize_row(flat[r], d, s, cpos, codes[r], norms[r:r + 1])
    return codes, norms


def query_f16(q_bf16: np.ndarray, seed: int = DEFAULT_SEED) -> np.ndarray:
    """T5: f16-rounded rotated query (as float64) for each bf16 row."""
    q = _c(q_bf16, np.uint16)
    d = q.shape[-1]
    flat = q.reshape(-1, d)
    out = np.empty(flat.shape, np.float64)
    for r in range(flat.shape[0]):
        _lib.uqo_query_f16(flat[r], d, seed, out[r])
    return out.reshape(q.shape)
