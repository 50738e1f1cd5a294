"""Host-detected errors on a real device: a slab larger than the GPU, a prompt
longer than the buffer, a misaligned query, key or value and a layer out of range are each
refused with a message, nothing is launched, and the context stays usable
(GPU; no fault is provoked)."""
import pytest
import torch

from decode_kv_cache_gb300 import longflow as lf

pytestmark = pytest.mark.gpu


def _small_step(cache):
    g = torch.Generator(device="cuda").manual_seed(3)
    b, hq, hkv, d = cache.batch, cache.q_heads, cache.kv_heads, cache.head_dim
    q = torch.randn(b, hq, d, generator=g, device="cuda").to(cache.dtype)
    k = torch.randn(b, hkv, d, generator=g, device="cuda").to(cache.dtype)
    v = torch.randn(b, hkv, d, generator=g, device="cuda").to(cache.dtype)
    out, ev = cache.decode_step(0, q, k, v)
    torch.cuda.synchronize()
    assert cache.check() == 0
    assert bool(torch.isfinite(out.float()).all())
    return out, ev


def test_slab_larger_than_the_device_is_refused():
    # The benchmark's per-layer shape (64 sequences, 8 KV heads, 3276 slots, which
    # has a launch shape) for 2000 layers: K alone is 2000 x 432 MB = 858 GB.
    with pytest.raises(lf.LFError, match="out of memory|does not fit"):
        lf.lf_cache_create_ex(2000, 64, 8, 32, 128, 3276, 64)
    # 8192 units of 16384 slots for 64 layers (4.4 TB): no tensor-core launch
    # shape fits, and the CUDA-core kernel's slab does not fit the device
    with pytest.raises(lf.LFError, match="out of memory|does not fit"):
        lf.lf_cache_create_ex(64, 1024, 8, 32, 128, 16384, 64)
    with lf.LFCache(1, 2, 2, 4, 128, 64, 4) as cache:   # the context still works
        _small_step(cache)


def test_bad_calls_are_refused_before_any_launch():
    with lf.LFCache(2, 2, 2, 4, 128, 64, 4) as cache:
        k = torch.zeros(2, 2, 80, 128, dtype=cache.dtype, device="cuda")
        with pytest.raises(lf.LFError, match="exceeds the buffer"):
            cache.prefill(0, k, k, [80, 10])
        n = 2 * 4 * 128
        q_mis = torch.zeros(n + 1, dtype=cache.dtype, device="cuda")[1:].view(2, 4, 128)
        kn = torch.zeros(2, 2, 128, dtype=cache.dtype, device="cuda")
        with pytest.raises(lf.LFError, match="16-byte aligned"):
            cache.decode_step(0, q_mis, kn, kn)
        m = 2 * 2 * 128
        kn_mis = torch.zeros(m + 1, dtype=cache.dtype, device="cuda")[1:].view(2, 2, 128)
        q = torch.zeros(2, 4, 128, dtype=cache.dtype, device="cuda")
        with pytest.raises(lf.LFError, match="16-byte aligned"):
            cache.decode_step(0, q, kn_mis, kn)
        with pytest.raises(lf.LFError, match="16-byte aligned"):
            cache.decode_step(0, q, kn, kn_mis)
        with pytest.raises(lf.LFError, match="outside"):
            cache.decode_step(2, torch.zeros(2, 4, 128, dtype=cache.dtype, device="cuda"), kn, kn)
        # nothing was written by the refused calls; a normal step still works
        views = cache.views()
        assert int(views["count"].sum()) == 0
        _small_step(cache)
        assert views["count"][0].tolist() == [[1, 1], [1, 1]]
