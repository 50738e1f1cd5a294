"""A layer too large for the tensor-core kernel's launch shape: the library
takes the CUDA-core kernel instead of refusing (GPU).

576 sequences x 8 KV heads of 16384 slots (38.7 GB of K and V): at 16384 slots
per unit only 16-CTA clusters fit the tensor-core kernel's per-CTA buffers,
9 of them are resident, and 4608 units would need 512+ items per cluster's
table.  The CUDA-core kernel runs one cluster per unit, with no such table."""
import math

import numpy as np
import pytest
import torch

from decode_kv_cache_gb300 import longflow as lf
from oracle.longflow_oracle import attention

pytestmark = pytest.mark.gpu


def test_very_large_layer_takes_the_cuda_core_kernel():
    B, HKV, HQ, D, CAP, W, P = 576, 8, 32, 128, 16384, 64, 32
    free, _ = torch.cuda.mem_get_info()
    if free < 48e9:
        pytest.skip("needs ~40 GB of free device memory")
    g = torch.Generator(device="cuda").manual_seed(21)
    with lf.LFCache(1, B, HKV, HQ, D, CAP, W) as cache:
        assert cache.layout.kernel == lf.LF_KERNEL_SIMT
        k = torch.randn(B, HKV, P, D, generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn(B, HKV, P, D, generator=g, device="cuda").to(torch.bfloat16)
        cache.prefill(0, k, v, [P] * B)
        q = torch.randn(B, HQ, D, generator=g, device="cuda").to(torch.bfloat16)
        kn = torch.randn(B, HKV, D, generator=g, device="cuda").to(torch.bfloat16)
        vn = torch.randn(B, HKV, D, generator=g, device="cuda").to(torch.bfloat16)
        out, ev = cache.decode_step(0, q, kn, vn)
        torch.cuda.synchronize()
        assert cache.check() == 0
        # not full: the new token is appended, nothing is evicted
        assert bool((ev == -1).all())
        assert cache.views()["count"][0].eq(P + 1).all()
        G = HQ // HKV
        for b, h in ((0, 0), (287, 5), (575, 7)):
            keys = torch.cat([k[b, h], kn[b, h][None]]).double().cpu().numpy()
            vals = torch.cat([v[b, h], vn[b, h][None]]).double().cpu().numpy()
            qq = q[b, h * G:(h + 1) * G].double().cpu().numpy()
            _, ref = attention(qq, keys, vals, 1.0 / math.sqrt(D))
            got = out[b, h * G:(h + 1) * G].double().cpu().numpy()
            # bf16 output: one rounding of values of magnitude < ~1
            np.testing.assert_allclose(got, ref, rtol=0, atol=1.6e-2)
