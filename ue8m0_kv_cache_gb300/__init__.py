"""Python binding of libuq.so: a paged FP4 E2M1 + UE8M0 KV cache ("UltraQuant")
for GB300, with FP8-E4M3 and BF16 caches of the same shape as anchors.

This module only marshals arguments: torch tensors in, raw device pointers and
sizes out to the C ABI declared in include/uq.h.  Every step of the path runs
in the library's CUDA kernels; there is no fallback.  Importing the module
fails if libuq.so has not been built (``python -m ue8m0_kv_cache_gb300.build``).
"""
import ctypes as C
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libuq.so")
if not os.path.exists(LIB_PATH):
    raise ImportError("libuq.so is not built (run python -m ue8m0_kv_cache_gb300.build): %s" % LIB_PATH)
_lib = C.CDLL(LIB_PATH)

UQ_OK = 0
FP4_UE8M0, FP8_E4M3, BF16, TQ4 = 0, 1, 2, 3
IN_BF16, IN_FP32 = 0, 1
DEFAULT_SEED = 42
STATUS_NAMES = {0: "UQ_OK", 1: "UQ_ERR_INVALID_ARG", 2: "UQ_ERR_UNSUPPORTED", 3: "UQ_ERR_ALIGNMENT",
                4: "UQ_ERR_WORKSPACE", 5: "UQ_ERR_CUDA", 6: "UQ_ERR_DEVICE_TIMEOUT", 7: "UQ_ERR_DEVICE_BOUNDS"}


class UqError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__("%s returned %s" % (where, STATUS_NAMES.get(status, status)))
        self.status = status


class UqCacheStruct(C.Structure):
    """Mirror of struct uq_cache."""
    _fields_ = [("dtype", C.c_int32), ("num_pages", C.c_int32), ("num_kv_heads", C.c_int32),
                ("page_size", C.c_int32), ("head_dim", C.c_int32),
                ("k_codes", C.c_void_p), ("k_scales", C.c_void_p), ("v_codes", C.c_void_p),
                ("v_scales", C.c_void_p), ("k_scale", C.c_float), ("v_scale", C.c_float),
                ("rot_seed", C.c_uint64), ("fp4_c", C.c_float)]


_vp, _i32, _i64, _f32, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t
_CP = C.POINTER(UqCacheStruct)
_sig = {
    "uq_cache_bytes": (_sz, [_CP, _i32]),
    "uq_quantize_append": (C.c_int, [_vp, _vp, _i32, _i64, _vp, _i32, _vp, _CP, _vp]),
    "uq_decode_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "uq_decode_attention": (C.c_int, [_vp, _CP, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "uq_decode_attention_fp8": (C.c_int, [_vp, _CP, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "uq_decode_attention_bf16": (C.c_int, [_vp, _CP, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "uq_decode_attention_tq4": (C.c_int, [_vp, _CP, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "uq_tq_codebook": (C.c_int, [_i32, _i32, _vp, _vp]),
    "uq_prefill_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "uq_prefill_attention": (C.c_int, [_vp, _vp, _i32, _CP, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "uq_calibrate_c": (C.c_int, [_vp, _i32, _i64, _i32, C.c_uint64, _vp, _i32, _i32, _vp, _vp]),
    "uq_cascade_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "uq_cascade_decode_attention": (C.c_int, [_vp, _CP, _vp, _i32, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _i32, _f32,
                                              _vp, _vp, _sz, _vp]),
    "uq_decode_attention_noalloc": (C.c_int, [_vp, _CP, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _vp]),
    "uq_decode_attention_append": (C.c_int, [_vp, _vp, _vp, _i32, _vp, _CP, _vp, _i32, _vp, _i32, _i32, _f32, _vp,
                                             _vp, _sz, _vp]),
    "uq_check_device_status": (C.c_int, [_vp]),
    "uq_status_string": (C.c_char_p, [C.c_int]),
    "uq_rotation_signs": (None, [C.c_uint64, _i32, _vp]),
    "uq_test_rotate": (C.c_int, [_vp, _i64, _i32, C.c_uint64, _i32, _vp, _vp]),
    "uq_test_quantize_rotated": (C.c_int, [_vp, _i64, _i32, _vp, _vp, _vp]),
    "uq_test_query_fp8": (C.c_int, [_vp, _i64, _i32, C.c_uint64, _vp, _vp]),
    "uq_test_cvt_e4m3": (C.c_int, [_vp, _i64, _vp, _vp]),
    "uq_test_cvt_e2m1": (C.c_int, [_vp, _i64, _vp, _vp]),
    "uq_test_scale_byte": (C.c_int, [_vp, _i64, _vp, _vp]),
    "uq_test_arm_decode_timeout": (C.c_int, [_i32, _i64]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = sorted(_sig)


def _check(status: int, where: str):
    if status != UQ_OK:
        raise UqError(status, where)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype, name):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))


class KVCache:
    """Device memory of one paged cache (torch tensors) plus its uq_cache struct."""

    def __init__(self, dtype: int, num_pages: int, num_kv_heads: int, page_size: int, head_dim: int,
                 device="cuda", rot_seed: int = DEFAULT_SEED, k_scale: float = 1.0, v_scale: float = 1.0,
                 fill: Optional[int] = None, fp4_c: float = 0.0):
        """fp4_c: the constant c of the FP4 scale rule (0: the default 0.156)."""
        self.dtype, self.num_pages, self.num_kv_heads = dtype, num_pages, num_kv_heads
        self.page_size, self.head_dim = page_size, head_dim
        shape = (num_pages, num_kv_heads, page_size)
        alloc = torch.empty if fill is None else (lambda *a, **k: torch.full(*a, fill, **k))
        if dtype == FP4_UE8M0:
            self.k_codes = alloc(shape + (head_dim // 2,), dtype=torch.uint8, device=device)
            self.v_codes = alloc(shape + (head_dim // 2,), dtype=torch.uint8, device=device)
            self.k_scales = alloc(shape + (head_dim // 32,), dtype=torch.uint8, device=device)
            self.v_scales = alloc(shape + (head_dim // 32,), dtype=torch.uint8, device=device)
        elif dtype == TQ4:
            self.k_codes = alloc(shape + (head_dim // 2,), dtype=torch.uint8, device=device)
            self.v_codes = alloc(shape + (head_dim // 2,), dtype=torch.uint8, device=device)
            nshape = shape + (4,)  # fp32 norm per row, held as 4 bytes
            self.k_scales = alloc(nshape, dtype=torch.uint8, device=device)
            self.v_scales = alloc(nshape, dtype=torch.uint8, device=device)
        else:
            el = torch.uint8 if dtype == FP8_E4M3 else torch.bfloat16
            if fill is None or dtype == FP8_E4M3:
                self.k_codes = alloc(shape + (head_dim,), dtype=el, device=device)
                self.v_codes = alloc(shape + (head_dim,), dtype=el, device=device)
            else:
                self.k_codes = torch.full(shape + (head_dim,), fill, dtype=torch.int16, device=device).view(el)
                self.v_codes = torch.full(shape + (head_dim,), fill, dtype=torch.int16, device=device).view(el)
            self.k_scales = self.v_scales = None
        self.struct = UqCacheStruct(dtype, num_pages, num_kv_heads, page_size, head_dim,
                                    _ptr(self.k_codes), _ptr(self.k_scales), _ptr(self.v_codes),
                                    _ptr(self.v_scales), k_scale, v_scale, rot_seed, fp4_c)

    @property
    def rot_seed(self) -> int:
        return self.struct.rot_seed

    def nbytes(self) -> int:
        return sum(uq_cache_bytes(self, w) for w in range(4))


def uq_cache_bytes(cache: KVCache, which: int) -> int:
    return int(_lib.uq_cache_bytes(C.byref(cache.struct), which))


def uq_quantize_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, cache: KVCache,
                       block_table: Optional[torch.Tensor] = None, stream=None) -> None:
    """Quantize-append k, v [T][Hkv][D] (bf16 or fp32) into `cache` at slot_mapping [T] (int64)."""
    if k.dtype not in (torch.bfloat16, torch.float32) or v.dtype != k.dtype:
        raise ValueError("k, v must both be bf16 or fp32")
    for t, n in ((k, "k"), (v, "v")):
        _need(t, k.dtype, n)
    _need(slot_mapping, torch.int64, "slot_mapping")
    T = k.shape[0]
    if tuple(k.shape) != (T, cache.num_kv_heads, cache.head_dim) or v.shape != k.shape or slot_mapping.numel() != T:
        raise ValueError("shape mismatch")
    mp = 0 if block_table is None else block_table.shape[-1]
    _check(_lib.uq_quantize_append(_ptr(k), _ptr(v), IN_FP32 if k.dtype == torch.float32 else IN_BF16, T,
                                   _ptr(block_table), mp, _ptr(slot_mapping), C.byref(cache.struct),
                                   _stream(stream)), "uq_quantize_append")


def uq_decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(_lib.uq_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim))


def workspace(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, device="cuda") -> torch.Tensor:
    n = uq_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def _decode(fn, name, q, cache, block_table, seq_lens, out, ws, sm_scale, stream):
    _need(q, torch.bfloat16, "q")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, D = q.shape
    if D != cache.head_dim or block_table.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out")
    if ws is None:
        ws = workspace(B, Hq, cache.num_kv_heads, D, q.device)
    _check(fn(_ptr(q), C.byref(cache.struct), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, Hq,
              float(sm_scale), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), name)
    return out


def uq_decode_attention(q, cache, block_table, seq_lens, out=None, workspace=None, sm_scale=0.0, stream=None):
    """Decode attention of q [B][Hq][D] bf16 over `cache`; returns fp32 [B][Hq][D]."""
    return _decode(_lib.uq_decode_attention, "uq_decode_attention", q, cache, block_table, seq_lens, out,
                   workspace, sm_scale, stream)


def uq_decode_attention_append(q, k_new, v_new, new_slots, cache, block_table, seq_lens, out=None, workspace=None,
                               sm_scale=0.0, stream=None):
    """One decode step: append each sequence's new token (k_new, v_new [B][Hkv][D], bf16 or fp32) at
    new_slots [B] (int64, -1 = none), then decode attention over seq_lens (which count the new token)."""
    if k_new.dtype not in (torch.bfloat16, torch.float32) or v_new.dtype != k_new.dtype:
        raise ValueError("k_new, v_new must both be bf16 or fp32")
    _need(k_new, k_new.dtype, "k_new")
    _need(v_new, k_new.dtype, "v_new")
    _need(new_slots, torch.int64, "new_slots")
    _need(q, torch.bfloat16, "q")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, D = q.shape
    if (tuple(k_new.shape) != (B, cache.num_kv_heads, cache.head_dim) or v_new.shape != k_new.shape
            or new_slots.numel() != B or D != cache.head_dim or block_table.shape[0] != B or seq_lens.numel() != B):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out")
    ws = workspace if workspace is not None else globals()["workspace"](B, Hq, cache.num_kv_heads, D, q.device)
    _check(_lib.uq_decode_attention_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), IN_FP32 if k_new.dtype == torch.float32 else IN_BF16, _ptr(new_slots),
        C.byref(cache.struct), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, Hq, float(sm_scale),
        _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "uq_decode_attention_append")
    return out


def uq_decode_attention_fp8(q, cache, block_table, seq_lens, out=None, workspace=None, sm_scale=0.0, stream=None):
    return _decode(_lib.uq_decode_attention_fp8, "uq_decode_attention_fp8", q, cache, block_table, seq_lens,
                   out, workspace, sm_scale, stream)


def uq_decode_attention_bf16(q, cache, block_table, seq_lens, out=None, workspace=None, sm_scale=0.0,
                             stream=None):
    return _decode(_lib.uq_decode_attention_bf16, "uq_decode_attention_bf16", q, cache, block_table, seq_lens,
                   out, workspace, sm_scale, stream)


def uq_decode_attention_tq4(q, cache, block_table, seq_lens, out=None, workspace=None, sm_scale=0.0, stream=None):
    return _decode(_lib.uq_decode_attention_tq4, "uq_decode_attention_tq4", q, cache, block_table, seq_lens, out,
                   workspace, sm_scale, stream)


def uq_tq_codebook(head_dim: int, bits: int = 4):
    """The TQ4 codebook the library uses: (f16 magnitudes of the non-negative
    half, ascending; fp32 decision thresholds, ascending) as float32 numpy arrays."""
    import numpy as np
    mags = np.zeros(1 << (bits - 1), np.float32)
    thr = np.zeros((1 << bits) - 1, np.float32)
    _check(_lib.uq_tq_codebook(head_dim, bits, mags.ctypes.data, thr.ctypes.data), "uq_tq_codebook")
    return mags, thr


def uq_prefill_workspace_bytes(num_q_tokens: int, batch: int, num_q_heads: int, num_kv_heads: int,
                               head_dim: int, max_keys: int) -> int:
    return int(_lib.uq_prefill_workspace_bytes(num_q_tokens, batch, num_q_heads, num_kv_heads, head_dim, max_keys))


def uq_prefill_attention(q, cu_q, cache, block_table, seq_lens, out=None, workspace=None, sm_scale=0.0,
                         stream=None):
    """Chunked-prefill attention: q [T][Hq][D] bf16, the chunk of sequence b in rows cu_q[b]..cu_q[b+1]-1
    (cu_q int32 [B+1]); seq_lens [B] count the chunk; returns fp32 [T][Hq][D]."""
    _need(q, torch.bfloat16, "q")
    _need(cu_q, torch.int32, "cu_q")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    T, Hq, D = q.shape
    B = seq_lens.numel()
    if D != cache.head_dim or cu_q.numel() != B + 1 or block_table.shape[0] != B:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out")
    if workspace is None:
        n = uq_prefill_workspace_bytes(T, B, Hq, cache.num_kv_heads, D, block_table.shape[1] * cache.page_size)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    _check(_lib.uq_prefill_attention(_ptr(q), _ptr(cu_q), T, C.byref(cache.struct), _ptr(block_table),
                                     block_table.shape[1], _ptr(seq_lens), B, Hq, float(sm_scale), _ptr(out),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)), "uq_prefill_attention")
    return out


def uq_cascade_workspace_bytes(batch: int, num_groups: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                               max_prefix_len: int) -> int:
    return int(_lib.uq_cascade_workspace_bytes(batch, num_groups, num_q_heads, num_kv_heads, head_dim,
                                               max_prefix_len))


def uq_cascade_decode_attention(q, cache, block_table, seq_lens, cu_seqs, prefix_lens, max_prefix_len, min_rows=128,
                                out=None, workspace=None, sm_scale=0.0, stream=None):
    """Cascade decode: q [B][Hq][D] bf16; group g = sequences cu_seqs[g]..cu_seqs[g+1]-1 (int32 [G+1]) whose first
    prefix_lens[g] keys (int32 [G]) are the same pages; returns fp32 [B][Hq][D], equal to uq_decode_attention."""
    _need(q, torch.bfloat16, "q")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(cu_seqs, torch.int32, "cu_seqs")
    _need(prefix_lens, torch.int32, "prefix_lens")
    B, Hq, D = q.shape
    ng = prefix_lens.numel()
    if D != cache.head_dim or seq_lens.numel() != B or block_table.shape[0] != B or cu_seqs.numel() != ng + 1:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out")
    if workspace is None:
        n = uq_cascade_workspace_bytes(B, ng, Hq, cache.num_kv_heads, D, max_prefix_len)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    _check(_lib.uq_cascade_decode_attention(_ptr(q), C.byref(cache.struct), _ptr(block_table), block_table.shape[1],
                                            _ptr(seq_lens), B, Hq, _ptr(cu_seqs), _ptr(prefix_lens), ng,
                                            int(max_prefix_len), int(min_rows), float(sm_scale), _ptr(out),
                                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                                            _stream(stream)), "uq_cascade_decode_attention")
    return out


def uq_calibrate_c(x: torch.Tensor, c_list, mode: int = 0, rot_seed: int = DEFAULT_SEED, stream=None):
    """Mean squared error of the FP4 round trip of the rotated rows of x ([N][D] bf16 or fp32) for each
    constant c of c_list (mode 0: the deployed power-of-two scale; -1: continuous scale c * absmax)."""
    if x.dtype not in (torch.bfloat16, torch.float32) or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA bf16 or fp32 tensor")
    d = x.shape[-1]
    n = x.numel() // d
    cs = (C.c_float * len(c_list))(*[float(c) for c in c_list])
    sse = torch.empty(len(c_list), dtype=torch.float64, device=x.device)
    _check(_lib.uq_calibrate_c(_ptr(x), IN_FP32 if x.dtype == torch.float32 else IN_BF16, n, d, rot_seed,
                               C.cast(cs, C.c_void_p), len(c_list), mode, _ptr(sse), _stream(stream)),
           "uq_calibrate_c")
    return (sse / max(1, n * d)).cpu().numpy()


def uq_check_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(_lib.uq_check_device_status(_stream(stream)))


def uq_status_string(status: int) -> str:
    return _lib.uq_status_string(status).decode()


def uq_rotation_signs(seed: int, d: int):
    buf = (C.c_int8 * d)()
    _lib.uq_rotation_signs(seed, d, C.cast(buf, C.c_void_p))
    return list(buf)


def uq_test_rotate(x: torch.Tensor, seed: int = DEFAULT_SEED, inverse: bool = False, stream=None) -> torch.Tensor:
    _need(x, torch.float32, "x")
    y = torch.empty_like(x)
    d = x.shape[-1]
    _check(_lib.uq_test_rotate(_ptr(x), x.numel() // d, d, seed, int(inverse), _ptr(y), _stream(stream)),
           "uq_test_rotate")
    return y


def uq_test_quantize_rotated(y: torch.Tensor, stream=None):
    _need(y, torch.float32, "y")
    d = y.shape[-1]
    n = y.numel() // d
    codes = torch.empty(y.shape[:-1] + (d // 2,), dtype=torch.uint8, device=y.device)
    scales = torch.empty(y.shape[:-1] + (d // 32,), dtype=torch.uint8, device=y.device)
    _check(_lib.uq_test_quantize_rotated(_ptr(y), n, d, _ptr(codes), _ptr(scales), _stream(stream)),
           "uq_test_quantize_rotated")
    return codes, scales


def uq_test_query_fp8(q: torch.Tensor, seed: int = DEFAULT_SEED, stream=None) -> torch.Tensor:
    _need(q, torch.bfloat16, "q")
    d = q.shape[-1]
    out = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    _check(_lib.uq_test_query_fp8(_ptr(q), q.numel() // d, d, seed, _ptr(out), _stream(stream)),
           "uq_test_query_fp8")
    return out


def uq_test_cvt_e2m1(r: torch.Tensor, stream=None) -> torch.Tensor:
    """E2M1 code (uint8, low nibble) of each fp32 value (even count)."""
    _need(r, torch.float32, "r")
    out = torch.empty(r.shape, dtype=torch.uint8, device=r.device)
    _check(_lib.uq_test_cvt_e2m1(_ptr(r), r.numel(), _ptr(out), _stream(stream)), "uq_test_cvt_e2m1")
    return out


def uq_test_scale_byte(m: torch.Tensor, stream=None) -> torch.Tensor:
    """UE8M0 scale byte of a group with absolute maximum |m| for each fp32 value."""
    _need(m, torch.float32, "m")
    out = torch.empty(m.shape, dtype=torch.uint8, device=m.device)
    _check(_lib.uq_test_scale_byte(_ptr(m), m.numel(), _ptr(out), _stream(stream)), "uq_test_scale_byte")
    return out


def uq_test_arm_decode_timeout(cta: int, budget_cycles: int) -> None:
    """Arm an injected timeout in the next warp-level decode launch (see uq.h):
    that call then ends with UQ_ERR_DEVICE_TIMEOUT in the device status word."""
    _check(_lib.uq_test_arm_decode_timeout(int(cta), int(budget_cycles)), "uq_test_arm_decode_timeout")


def uq_test_cvt_e4m3(x: torch.Tensor, stream=None) -> torch.Tensor:
    _need(x, torch.float32, "x")
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(_lib.uq_test_cvt_e4m3(_ptr(x), x.numel(), _ptr(out), _stream(stream)), "uq_test_cvt_e4m3")
    return out
