"""lf_prefill_fill_noalloc: the prefill entry point for callers that cannot
allocate device memory (an engine that hands out slices of its own
pre-reserved pool, code where an allocation's implicit synchronisation is not
allowed).  Such a caller owns the slab; the entry point moves the prompt
lengths to the GPU through a fixed array built into the library.

The test fills caller-owned buffers with the no-allocation entry point and a
library-owned cache with lf_prefill_fill, from the same inputs, and requires
the two slabs to agree -- on two calls in a row, the second with different
(shorter) prompts so that stale contents of the shared array would show.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import pytest
import torch

from decode_kv_cache_gb300 import longflow as lf

pytestmark = pytest.mark.gpu


def _caller_owned_slab(cache):
    """Buffers with the cache's layout, allocated by the caller (torch here)."""
    lay = cache.layout
    L, b, g, s, d = lay.layers, lay.batch, lay.kv_heads, lay.slot_stride, lay.head_dim
    own = {
        "k": torch.zeros(L, b, g, s, d, dtype=cache.dtype, device="cuda"),
        "v": torch.zeros(L, b, g, s, d, dtype=cache.dtype, device="cuda"),
        "vnorm": torch.zeros(L, b, g, s, dtype=torch.float32, device="cuda"),
        "pos": torch.full((L, b, g, s), -1, dtype=torch.int32, device="cuda"),
        "count": torch.zeros(L, b, g, dtype=torch.int32, device="cuda"),
        "next_pos": torch.zeros(L, b, g, dtype=torch.int32, device="cuda"),
    }
    dst = lf.LFLayout()
    for name in ("layers", "batch", "kv_heads", "q_heads", "head_dim", "capacity", "slot_stride",
                 "window", "dtype", "evict"):
        setattr(dst, name, getattr(lay, name))
    for name, t in own.items():
        setattr(dst, name, t.data_ptr())
    return dst, own


@pytest.mark.parametrize("dtype,head_dim", [("bf16", 128), ("f32", 16)])
def test_noalloc_prefill_matches_prefill_fill(dtype, head_dim):
    layers, batch, kv_heads, q_heads, capacity, window = 2, 3, 2, 4, 40, 4
    cache = lf.LFCache(layers, batch, kv_heads, q_heads, head_dim, capacity, window, dtype=dtype)
    try:
        dst, own = _caller_owned_slab(cache)
        lib_slab = cache.views()
        g = torch.Generator(device="cuda").manual_seed(7)
        for lens in ([37, 12, 40], [5, 33, 0]):
            pmax = max(lens)
            k = torch.randn(batch, kv_heads, pmax, head_dim, generator=g, device="cuda").to(cache.dtype)
            v = torch.randn(batch, kv_heads, pmax, head_dim, generator=g, device="cuda").to(cache.dtype)
            cache.prefill(1, k, v, lens)                          # existing entry point
            lf.lf_prefill_fill_noalloc(dst, 1, k, v, lens, pmax)  # no allocation
            torch.cuda.synchronize()
            for name in ("k", "v", "pos", "count", "next_pos"):
                assert torch.equal(own[name][1], lib_slab[name][1]), name
            # same arithmetic on both paths: the fp32 norms agree exactly
            torch.testing.assert_close(own["vnorm"][1], lib_slab["vnorm"][1], rtol=0, atol=0)
            # the other layer is untouched
            assert int(own["count"][0].abs().sum()) == 0
        # batches beyond the fixed array are refused
        big = lf.LFLayout.from_buffer_copy(dst)
        big.batch = 16385
        with pytest.raises(lf.LFError, match="LF_NOALLOC_MAX_BATCH"):
            lf.lf_prefill_fill_noalloc(big, 0, None, None, [0] * 16385, 0)
    finally:
        cache.close()
