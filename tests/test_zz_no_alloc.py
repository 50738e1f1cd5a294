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
    """Buffers with the cache's layout, allocated by the caller (torch here).
    The H2O accumulators and the deferred choice start at values the prefill
    must overwrite."""
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
    if lay.acc:
        own["acc"] = torch.full((L, b, g, s), 3.0, dtype=torch.float32, device="cuda")
    if lay.pending:
        own["pending"] = torch.full((L, b, g), 7, dtype=torch.int32, device="cuda")
    dst = lf.LFLayout()
    for name in ("layers", "batch", "kv_heads", "q_heads", "head_dim", "capacity", "slot_stride",
                 "window", "dtype", "evict", "norm"):
        setattr(dst, name, getattr(lay, name))
    for name, t in own.items():
        setattr(dst, name, t.data_ptr())
    return dst, own


POLICIES = {
    "default": ({}, ([37, 12, 40], [5, 33, 0])),
    "h2o_l2": (dict(score="h2o", norm=2), ([37, 12, 40], [5, 33, 0])),
    # deferred: a prompt leaves one slot free
    "deferred": (dict(deferred=True), ([37, 12, 39], [5, 33, 0])),
}


@pytest.mark.parametrize("policy", sorted(POLICIES))
@pytest.mark.parametrize("dtype,head_dim", [("bf16", 128), ("f32", 16)])
def test_noalloc_prefill_matches_prefill_fill(dtype, head_dim, policy):
    layers, batch, kv_heads, q_heads, capacity, window = 2, 3, 2, 4, 40, 4
    kw, prompts = POLICIES[policy]
    cache = lf.LFCache(layers, batch, kv_heads, q_heads, head_dim, capacity, window, dtype=dtype,
                       **kw)
    try:
        dst, own = _caller_owned_slab(cache)
        assert ("acc" in own) == (kw.get("score") == "h2o")
        assert ("pending" in own) == bool(kw.get("deferred"))
        lib_slab = cache.views()
        g = torch.Generator(device="cuda").manual_seed(7)
        for lens in prompts:
            pmax = max(lens)
            k = torch.randn(batch, kv_heads, pmax, head_dim, generator=g, device="cuda").to(cache.dtype)
            v = torch.randn(batch, kv_heads, pmax, head_dim, generator=g, device="cuda").to(cache.dtype)
            cache.prefill(1, k, v, lens)                          # existing entry point
            lf.lf_prefill_fill_noalloc(dst, 1, k, v, lens, pmax)  # no allocation
            assert lf.lf_last_status() == lf.LF_OK                # a success leaves no failure
            torch.cuda.synchronize()
            for name in ("k", "v", "pos", "count", "next_pos", "pending"):
                if name in own:
                    assert torch.equal(own[name][1], lib_slab[name][1]), name
            # same arithmetic on both paths: the fp32 norms agree exactly
            torch.testing.assert_close(own["vnorm"][1], lib_slab["vnorm"][1], rtol=0, atol=0)
            if "acc" in own:
                assert torch.equal(own["acc"][1], lib_slab["acc"][1])
                assert int(torch.count_nonzero(own["acc"][1])) == 0
            if "pending" in own:
                assert bool((own["pending"][1] == -1).all())
            # the other layer is untouched
            assert int(own["count"][0].abs().sum()) == 0
        if kw.get("deferred"):
            # a deferred buffer filled by its prompt would have no slot chosen
            with pytest.raises(lf.LFError, match="deferred"):
                lf.lf_prefill_fill_noalloc(dst, 1, k, v, [capacity, 0, 0], capacity)
        # batches beyond the fixed array are refused ...
        big = lf.LFLayout.from_buffer_copy(dst)
        big.batch = 16385
        with pytest.raises(lf.LFError, match="LF_NOALLOC_MAX_BATCH"):
            lf.lf_prefill_fill_noalloc(big, 0, None, None, [0] * 16385, 0)
        assert lf.lf_last_status() == lf.LF_ERR_ARG
        # ... and the next successful call clears that failure
        lf.lf_prefill_fill_noalloc(dst, 0, k, v, [1, 0, 2], pmax)
        assert lf.lf_last_status() == lf.LF_OK and lf.lf_last_error() == ""
        torch.cuda.synchronize()
        assert own["count"][0].flatten().tolist() == [1, 1, 0, 0, 2, 2]
    finally:
        cache.close()
