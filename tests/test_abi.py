"""The C-ABI library loads and exports every symbol include/longflow.h declares;
host-side argument checks answer without touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from decode_kv_cache_gb300 import longflow as lf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "longflow.h")


@pytest.fixture(scope="module")
def lib():
    from decode_kv_cache_gb300 import build as b
    b.build()
    return lf.load_library()


def _header():
    return open(HEADER).read()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", _header(), flags=re.S)
    return sorted(set(re.findall(r"\b(lf_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["lf_cache_create", "lf_cache_create_ex", "lf_prefill_fill", "lf_decode_step",
                     "lf_cache_destroy", "lf_cache_check", "lf_cache_layout", "lf_last_error"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in longflow.h but not exported"


def test_abi_version_matches_header(lib):
    m = re.search(r"#define LF_ABI_VERSION (\d+)", _header())
    assert lf.lf_abi_version() == int(m.group(1))


def test_constants_match_header():
    text = _header()
    for name in ["LF_OK", "LF_ERR_ARG", "LF_ERR_OOM", "LF_ERR_CUDA", "LF_ERR_DEVICE",
                 "LF_ERR_UNSUPPORTED", "LF_BF16", "LF_F32", "LF_KERNEL_AUTO", "LF_KERNEL_SIMT",
                 "LF_KERNEL_TENSOR_CORE", "LF_SCORE_LONGFLOW", "LF_SCORE_H2O", "LF_SCOPE_KV_HEAD",
                 "LF_SCOPE_LAYER", "LF_EVICT_OFF", "LF_EVICT_LONGFLOW", "LF_EVICT_RKV"]:
        m = re.search(rf"\b{name}\s*=\s*(-?\d+)", text)
        assert m and int(m.group(1)) == getattr(lf, name), name
    for name in ["LF_DEVERR_NONFINITE", "LF_DEVERR_STATE", "LF_DEVERR_TIMEOUT"]:
        m = re.search(rf"#define {name} (\d+)", text)
        assert m and int(m.group(1)) == getattr(lf, name), name


def test_header_is_plain_c_and_structs_match_binding(tmp_path):
    """Compile the header as C11 with gcc; sizes and field offsets of the
    structs must equal the ctypes mirrors."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    fields_cfg = [f for f, _ in lf.LFConfig._fields_]
    fields_lay = [f for f, _ in lf.LFLayout._fields_]
    src = tmp_path / "sizes.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "longflow.h"', 'int main(void){',
             'printf("%zu %zu\\n", sizeof(lf_config), sizeof(lf_layout));']
    for f in fields_cfg:
        lines.append(f'printf("%zu ", offsetof(lf_config, {f}));')
    lines.append('printf("\\n");')
    for f in fields_lay:
        lines.append(f'printf("%zu ", offsetof(lf_layout, {f}));')
    lines.append('printf("\\n"); return 0; }')
    src.write_text("\n".join(lines))
    exe = tmp_path / "sizes"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    sz_cfg, sz_lay = map(int, out[0].split())
    assert sz_cfg == ctypes.sizeof(lf.LFConfig)
    assert sz_lay == ctypes.sizeof(lf.LFLayout)
    assert [int(x) for x in out[1].split()] == [getattr(lf.LFConfig, f).offset for f in fields_cfg]
    assert [int(x) for x in out[2].split()] == [getattr(lf.LFLayout, f).offset for f in fields_lay]


@pytest.mark.parametrize("args,msg", [
    ((1, 1, 3, 4, 128, 64, 4), "multiple of kv_heads"),
    ((0, 1, 1, 1, 128, 64, 4), ">= 1"),
    ((1, 1, 1, 1, 128, 64, -1), "window >= 0"),
    ((1, 1, 8, 32, 96, 64, 4), "no kernel for head_dim 96"),
    ((1, 1, 2, 6, 128, 64, 4), "group size 3"),
    ((1, 1, 1, 1, 128, 8, 8), "window + sinks (8 + 0) must be smaller"),
])
def test_argument_errors_need_no_gpu(lib, args, msg):
    h = lib.lf_cache_create(*args)
    assert not h
    assert msg in lf.lf_last_error()


def test_bad_config_fields(lib):
    with pytest.raises(lf.LFError, match="cluster"):
        lf.lf_cache_create_ex(1, 1, 1, 1, 128, 64, 4, cluster=3)
    with pytest.raises(lf.LFError, match="stages"):
        lf.lf_cache_create_ex(1, 1, 1, 1, 128, 64, 4, stages=1)
    with pytest.raises(lf.LFError, match="budget"):
        lf.lf_cache_create_ex(1, 2, 1, 1, 128, 64, 4, budgets=[64, 65])
    with pytest.raises(lf.LFError, match="window"):
        lf.lf_cache_create_ex(1, 2, 1, 1, 128, 64, 8, budgets=[64, 8])


def test_bad_policy_fields(lib):
    """The policy variants are checked on the host before any CUDA call."""
    with pytest.raises(lf.LFError, match="policy"):
        lf.lf_cache_create_ex(1, 1, 1, 1, 128, 64, 4, score=2)
    with pytest.raises(lf.LFError, match="policy"):
        lf.lf_cache_create_ex(1, 1, 1, 1, 128, 64, 4, norm=3)
    with pytest.raises(lf.LFError, match="policy"):
        lf.lf_cache_create_ex(1, 1, 1, 1, 128, 64, 4, sinks=-1)
    with pytest.raises(lf.LFError, match="policy"):
        lf.lf_cache_create_ex(1, 1, 1, 1, 128, 64, 4, scope=5)
    # the window and the sinks together must leave a candidate in every buffer
    with pytest.raises(lf.LFError, match=r"window \+ sinks \(4 \+ 4\)"):
        lf.lf_cache_create_ex(1, 2, 1, 1, 128, 64, 4, budgets=[64, 8], sinks=4)
    # deferred eviction protects the new token through the window
    with pytest.raises(lf.LFError, match="window >= 1"):
        lf.lf_cache_create_ex(1, 1, 1, 1, 128, 64, 0, deferred=True)


def test_bad_rkv_fields(lib):
    """R-KV mode: the compression kernel's limits are checked on the host."""
    with pytest.raises(lf.LFError, match="bf16, head_dim 128"):
        lf.lf_cache_create_ex(1, 1, 2, 8, 128, 400, 0, dtype="f32", evict="rkv")
    with pytest.raises(lf.LFError, match="no per-sequence budgets"):
        lf.lf_cache_create_ex(1, 2, 2, 8, 128, 400, 0, evict="rkv", budgets=[300, 300])
    with pytest.raises(lf.LFError, match="capacity <= 4096"):
        lf.lf_cache_create_ex(1, 1, 2, 8, 128, 5000, 0, evict="rkv")
    with pytest.raises(lf.LFError, match="alpha \\* group <= 64"):
        lf.lf_cache_create_ex(1, 1, 1, 8, 128, 400, 0, evict="rkv", rkv_alpha=9)
    with pytest.raises(lf.LFError, match="lambda and tau"):
        lf.lf_cache_create_ex(1, 1, 2, 8, 128, 400, 0, evict="rkv", rkv_lambda=1.5)
    with pytest.raises(lf.LFError, match="evict must be"):
        lf.lf_cache_create_ex(1, 1, 2, 8, 128, 400, 0, evict=3)
    assert lib.lf_rkv_compress(None, 0, None, None) == lf.LF_ERR_ARG


def test_null_handles(lib):
    assert lib.lf_cache_destroy(None) == lf.LF_OK
    assert lib.lf_decode_step(None, 0, None, None, None, None, None, None) == lf.LF_ERR_ARG
    assert lib.lf_prefill_fill(None, 0, None, None, None, 0, None) == lf.LF_ERR_ARG
    assert lib.lf_cache_layout(None, None) == lf.LF_ERR_ARG
    assert lib.lf_cache_check(None, None, None) == lf.LF_ERR_ARG
    assert lib.lf_launch_plan(None, 0, None, None, None, 0) == lf.LF_ERR_ARG


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = lib.lf_cache_create(1, 1, 1, 2, 16, 32, 4)
    assert not h
    assert lf.lf_last_error()  # a CUDA error message, no crash


def test_stored_traffic_needs_the_measured_kernel(tmp_path, monkeypatch):
    """bench.py reports the ncu traffic of the decode kernel only while the
    committed summary was measured on the current kernel sources."""
    import bench
    good = bench.stored_traffic("qwen3-8b-steady", 64)
    text = open(bench.PROFILE_SUMMARY).read()
    stale = tmp_path / "summary.md"
    stale.write_text(text.replace(bench.kernel_source_hash(), "0" * 64))
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(stale))
    assert bench.stored_traffic("qwen3-8b-steady", 64) is None
    assert good is None or good > 0
    assert bench.stored_traffic("ragged-serving", 64) is None


def test_last_status_tells_why_create_failed(lib):
    """lf_cache_create* returns NULL on failure; lf_last_status says why."""
    assert not lib.lf_cache_create(1, 1, 3, 4, 16, 32, 4)        # q_heads % kv_heads != 0
    assert lf.lf_last_status() == lf.LF_ERR_ARG
    with pytest.raises(lf.LFError) as e:
        lf.lf_cache_create(1, 1, 1, 2, 16, 32, 40)               # window >= budget
    assert e.value.code == lf.LF_ERR_ARG
    # a call that resets the message resets the status too
    assert lib.lf_cache_destroy(None) == lf.LF_OK
    assert lf.lf_last_status() == lf.LF_OK and lf.lf_last_error() == ""
    import torch
    if not torch.cuda.is_available():
        with pytest.raises(lf.LFError) as e:
            lf.lf_cache_create(1, 1, 1, 2, 16, 32, 4)           # valid, but no device here
        assert e.value.code == lf.LF_ERR_CUDA
