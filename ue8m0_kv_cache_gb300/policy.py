"""Per-layer precision policy and a multi-layer paged KV cache.

The UltraQuant pages deploy the 4-bit cache with boundary-layer protection: the
first two and the last two attention layers keep a BF16 KV cache, every other
layer uses the FP4 E2M1 + UE8M0 cache ("UltraQuant" review, manon006.tistory.com
/395, §4.1; "kv-cache-4bit-serving-residency-collapse", footnote 6).  They keep
one global shrink constant c = 0.156 and name per-layer constants and
sensitivity-driven mixed policies as the open options (review §7.3); a layer's
constant can be measured with uq_calibrate_c on its captured keys.

LayerPolicy says which cache format (and which c) each layer gets;
LayeredKVCache holds one library cache per layer on a shared page layout and
runs one decode step over all layers (append of the step's token, then decode
attention), eagerly or as a captured CUDA graph.  Every step of the data path
runs in the library's kernels; this module only routes calls.
"""
from typing import List, Optional, Sequence

import torch

from . import (BF16, FP4_UE8M0, FP8_E4M3, KVCache, uq_decode_attention, uq_decode_attention_append,
               uq_decode_attention_bf16, uq_decode_attention_fp8, uq_quantize_append, workspace)

_DECODE = {BF16: uq_decode_attention_bf16, FP8_E4M3: uq_decode_attention_fp8}


class LayerPolicy:
    """Cache format of each of num_layers attention layers.

    boundary: layers [0, boundary) and [num_layers - boundary, num_layers) use
    `edge` (BF16 by default, the pages' protection of the first and last two
    layers); the others use `inner` (FP4).  overrides: {layer: dtype} for a
    mixed policy from a sensitivity measurement.  fp4_c: one constant for all
    FP4 layers or a per-layer sequence (0 = the default 0.156)."""

    def __init__(self, num_layers: int, boundary: int = 2, inner: int = FP4_UE8M0, edge: int = BF16,
                 overrides: Optional[dict] = None, fp4_c=0.0):
        if num_layers < 1 or boundary < 0:
            raise ValueError("num_layers >= 1 and boundary >= 0 required")
        self.num_layers = num_layers
        self.dtypes = [edge if (l < boundary or l >= num_layers - boundary) else inner for l in range(num_layers)]
        for l, d in (overrides or {}).items():
            self.dtypes[l] = d
        if isinstance(fp4_c, (int, float)):
            self.c = [float(fp4_c)] * num_layers
        else:
            if len(fp4_c) != num_layers:
                raise ValueError("one constant per layer")
            self.c = [float(x) for x in fp4_c]

    def dtype(self, layer: int) -> int:
        return self.dtypes[layer]

    def fp4_c(self, layer: int) -> float:
        return self.c[layer] if self.dtypes[layer] == FP4_UE8M0 else 0.0

    def count(self, dtype: int) -> int:
        return sum(1 for d in self.dtypes if d == dtype)


class LayeredKVCache:
    """One paged cache per layer, all with the same page geometry (one block
    table serves every layer), formats from a LayerPolicy."""

    def __init__(self, policy: LayerPolicy, num_pages: int, num_kv_heads: int, page_size: int, head_dim: int,
                 device="cuda", rot_seed: Optional[int] = None, fill: Optional[int] = None):
        self.policy = policy
        kw = {} if rot_seed is None else {"rot_seed": rot_seed}
        self.layers: List[KVCache] = [
            KVCache(policy.dtype(l), num_pages, num_kv_heads, page_size, head_dim, device=device,
                    fp4_c=policy.fp4_c(l), fill=fill, **kw)
            for l in range(policy.num_layers)]
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        self._graph = None

    def __len__(self) -> int:
        return len(self.layers)

    def nbytes(self) -> int:
        return sum(c.nbytes() for c in self.layers)

    def append(self, layer: int, k: torch.Tensor, v: torch.Tensor, slots: torch.Tensor, stream=None):
        uq_quantize_append(k, v, slots, self.layers[layer], stream=stream)

    def decode(self, layer: int, q, block_table, seq_lens, out=None, ws=None, stream=None):
        c = self.layers[layer]
        fn = _DECODE.get(c.dtype, uq_decode_attention)
        return fn(q, c, block_table, seq_lens, out=out, workspace=ws, stream=stream)

    def decode_step(self, q: Sequence[torch.Tensor], k_new: Sequence[torch.Tensor], v_new: Sequence[torch.Tensor],
                    new_slots: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                    out: Sequence[torch.Tensor], ws: torch.Tensor, stream=None):
        """One decode step of every layer: each layer's new token (k_new[l], v_new[l] [B][Hkv][D]) is
        appended at new_slots, then q[l] attends over seq_lens (which count the new token).  FP4
        layers do both in one launch; the other formats append, then decode."""
        for l, c in enumerate(self.layers):
            if c.dtype == FP4_UE8M0:
                uq_decode_attention_append(q[l], k_new[l], v_new[l], new_slots, c, block_table, seq_lens,
                                           out=out[l], workspace=ws, stream=stream)
            else:
                uq_quantize_append(k_new[l], v_new[l], new_slots, c, stream=stream)
                self.decode(l, q[l], block_table, seq_lens, out=out[l], ws=ws, stream=stream)

    def capture_step(self, q, k_new, v_new, new_slots, block_table, seq_lens, out, ws):
        """Capture decode_step on these (static) buffers in a CUDA graph; replay() runs it.  Update the
        buffers in place between replays (seq_lens, new_slots, q, k_new, v_new)."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):  # one eager step first: per-device kernel setup happens outside capture
            self.decode_step(q, k_new, v_new, new_slots, block_table, seq_lens, out, ws, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.decode_step(q, k_new, v_new, new_slots, block_table, seq_lens, out, ws,
                             stream=torch.cuda.current_stream())
        self._graph = g
        return g

    def replay(self):
        if self._graph is None:
            raise RuntimeError("capture_step first")
        self._graph.replay()


def layered_workspace(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, device="cuda"):
    """One decode workspace serves every layer (the layers run in stream order)."""
    return workspace(batch, num_q_heads, num_kv_heads, head_dim, device)
