"""Thin Python binding of liblongflow.so (ctypes).

The functions below carry the C names and only marshal arguments: torch
tensors become device pointers, torch streams become ``cudaStream_t``.  Every
step of the decode path runs in the library's CUDA kernels; there is no
Python or CPU fallback, and a missing library raises immediately.

``LFCache`` is a convenience owner of one cache handle that checks tensor
shapes/dtypes before calling the C functions, and exposes the slab as torch
views (through ``__cuda_array_interface__``) for tests, snapshots and restores.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

__all__ = [
    "LF_OK", "LF_ERR_ARG", "LF_ERR_OOM", "LF_ERR_CUDA", "LF_ERR_DEVICE", "LF_ERR_UNSUPPORTED",
    "LF_BF16", "LF_F32", "LF_KERNEL_AUTO", "LF_KERNEL_SIMT", "LF_KERNEL_TENSOR_CORE",
    "LF_DEVERR_NONFINITE", "LF_DEVERR_STATE", "LF_DEVERR_TIMEOUT",
    "LF_EVICT_OFF", "LF_EVICT_LONGFLOW", "LF_EVICT_RKV", "LF_SCORE_LONGFLOW", "LF_SCORE_H2O",
    "LF_SCOPE_KV_HEAD", "LF_SCOPE_LAYER",
    "LFError", "LFConfig", "LFLayout", "load_library", "library_path",
    "lf_cache_create", "lf_cache_create_ex", "lf_cache_destroy", "lf_prefill_fill",
    "lf_decode_step", "lf_cache_check", "lf_cache_layout", "lf_last_error", "lf_last_status",
    "lf_abi_version",
    "lf_prefill_fill_noalloc", "lf_rkv_compress", "lf_launch_plan", "lf_launch_plan_for",
    "LFCache",
]

LF_OK, LF_ERR_ARG, LF_ERR_OOM, LF_ERR_CUDA, LF_ERR_DEVICE, LF_ERR_UNSUPPORTED = 0, -1, -2, -3, -5, -7
LF_BF16, LF_F32 = 0, 1
LF_KERNEL_AUTO, LF_KERNEL_SIMT, LF_KERNEL_TENSOR_CORE = 0, 1, 2
_KERNEL = {"auto": LF_KERNEL_AUTO, "simt": LF_KERNEL_SIMT, "tc": LF_KERNEL_TENSOR_CORE}
LF_EVICT_OFF, LF_EVICT_LONGFLOW, LF_EVICT_RKV = 0, 1, 2
_EVICT = {"off": LF_EVICT_OFF, "longflow": LF_EVICT_LONGFLOW, "rkv": LF_EVICT_RKV}
LF_SCORE_LONGFLOW, LF_SCORE_H2O = 0, 1
_SCORE = {"longflow": LF_SCORE_LONGFLOW, "h2o": LF_SCORE_H2O}
LF_SCOPE_KV_HEAD, LF_SCOPE_LAYER = 0, 1
_SCOPE = {"kv_head": LF_SCOPE_KV_HEAD, "layer": LF_SCOPE_LAYER}
LF_DEVERR_NONFINITE, LF_DEVERR_STATE, LF_DEVERR_TIMEOUT = 1, 2, 4

_DTYPE = {"bf16": LF_BF16, "f32": LF_F32}
_TORCH_DTYPE = {LF_BF16: torch.bfloat16, LF_F32: torch.float32}


class LFError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class LFConfig(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("evict", ctypes.c_int),
                ("budgets", ctypes.POINTER(ctypes.c_int32)), ("cluster", ctypes.c_int),
                ("stages", ctypes.c_int), ("kernel", ctypes.c_int),
                ("score", ctypes.c_int), ("norm", ctypes.c_int), ("sinks", ctypes.c_int),
                ("deferred", ctypes.c_int), ("scope", ctypes.c_int),
                ("rkv_buffer", ctypes.c_int), ("rkv_alpha", ctypes.c_int), ("rkv_beta", ctypes.c_int),
                ("rkv_lambda", ctypes.c_float), ("rkv_tau", ctypes.c_float)]


class LFLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "layers", "batch", "kv_heads", "q_heads", "head_dim", "capacity", "slot_stride",
        "window", "dtype", "evict", "cluster", "stages", "kernel")] + [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("vnorm", ctypes.c_void_p),
        ("pos", ctypes.c_void_p), ("count", ctypes.c_void_p), ("next_pos", ctypes.c_void_p),
        ("budget", ctypes.c_void_p), ("err", ctypes.c_void_p)] + [
        (n, ctypes.c_int) for n in ("score", "norm", "sinks", "deferred", "scope")] + [
        ("acc", ctypes.c_void_p), ("pending", ctypes.c_void_p)] + [
        (n, ctypes.c_int) for n in ("rkv_buffer", "rkv_alpha", "rkv_beta")] + [
        ("rkv_lambda", ctypes.c_float), ("rkv_tau", ctypes.c_float),
        ("split_units", ctypes.c_int), ("split_cnt", ctypes.c_void_p)]


_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return os.environ.get("LONGFLOW_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                          "liblongflow.so")


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load liblongflow.so once; raise if it is missing (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"liblongflow.so not found at {path}: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I, VP = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    lib.lf_cache_create.restype = P
    lib.lf_cache_create.argtypes = [I] * 7
    lib.lf_cache_create_ex.restype = P
    lib.lf_cache_create_ex.argtypes = [I] * 7 + [ctypes.POINTER(LFConfig)]
    lib.lf_cache_destroy.restype = I
    lib.lf_cache_destroy.argtypes = [P]
    lib.lf_prefill_fill.restype = I
    lib.lf_prefill_fill.argtypes = [P, I, VP, VP, ctypes.POINTER(ctypes.c_int32), I, VP]
    lib.lf_decode_step.restype = I
    lib.lf_decode_step.argtypes = [P, I, VP, VP, VP, VP, VP, VP]
    lib.lf_cache_check.restype = I
    lib.lf_cache_check.argtypes = [P, VP, ctypes.POINTER(ctypes.c_int32)]
    lib.lf_cache_layout.restype = I
    lib.lf_cache_layout.argtypes = [P, ctypes.POINTER(LFLayout)]
    lib.lf_last_error.restype = ctypes.c_char_p
    lib.lf_last_error.argtypes = []
    lib.lf_abi_version.restype = I
    lib.lf_abi_version.argtypes = []
    lib.lf_last_status.restype = I
    lib.lf_last_status.argtypes = []
    lib.lf_rkv_compress.restype = I
    lib.lf_rkv_compress.argtypes = [P, I, VP, VP]
    lib.lf_launch_plan.restype = I
    lib.lf_launch_plan.argtypes = [P, I] + [ctypes.POINTER(ctypes.c_int32)] * 3 + [I]
    lib.lf_launch_plan_for.restype = I
    lib.lf_launch_plan_for.argtypes = ([ctypes.POINTER(ctypes.c_int32)] + [I] * 4 +
                                       [ctypes.POINTER(ctypes.c_int32)] * 3)
    lib.lf_prefill_fill_noalloc.restype = I
    lib.lf_prefill_fill_noalloc.argtypes = [ctypes.POINTER(LFLayout), I, VP, VP,
                                            ctypes.POINTER(ctypes.c_int32), I, VP]
    _lib = lib
    return lib


# ---- C-named wrappers (argument marshalling only) ---------------------------

def lf_last_error() -> str:
    return (load_library().lf_last_error() or b"").decode()


def lf_last_status() -> int:
    return load_library().lf_last_status()


def _create_failed() -> "LFError":
    """The error of a create call that returned NULL, with the library's status."""
    return LFError(lf_last_status() or LF_ERR_ARG, lf_last_error())


def lf_abi_version() -> int:
    return load_library().lf_abi_version()


def _check(code: int) -> int:
    if code != LF_OK:
        raise LFError(code, lf_last_error())
    return code


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def lf_cache_create(layers, batch, kv_heads, q_heads, head_dim, budget, window) -> int:
    h = load_library().lf_cache_create(layers, batch, kv_heads, q_heads, head_dim, budget, window)
    if not h:
        raise _create_failed()
    return h


def lf_cache_create_ex(layers, batch, kv_heads, q_heads, head_dim, capacity, window,
                       dtype="bf16", evict=True, budgets: Optional[Sequence[int]] = None,
                       cluster=0, stages=0, kernel="auto", score="longflow", norm=1, sinks=0,
                       deferred=False, scope="kv_head", rkv_buffer=0, rkv_alpha=0, rkv_beta=0,
                       rkv_lambda=0.0, rkv_tau=0.0) -> int:
    cfg = LFConfig()
    cfg.dtype = _DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    cfg.evict = _EVICT[evict] if isinstance(evict, str) else int(evict)
    arr = None
    if budgets is not None:
        arr = (ctypes.c_int32 * len(budgets))(*[int(x) for x in budgets])
        cfg.budgets = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
    cfg.cluster = int(cluster)
    cfg.stages = int(stages)
    cfg.kernel = _KERNEL[kernel] if isinstance(kernel, str) else int(kernel)
    cfg.score = _SCORE[score] if isinstance(score, str) else int(score)
    cfg.norm = int(norm)
    cfg.sinks = int(sinks)
    cfg.deferred = int(bool(deferred))
    cfg.scope = _SCOPE[scope] if isinstance(scope, str) else int(scope)
    cfg.rkv_buffer, cfg.rkv_alpha, cfg.rkv_beta = int(rkv_buffer), int(rkv_alpha), int(rkv_beta)
    cfg.rkv_lambda, cfg.rkv_tau = float(rkv_lambda), float(rkv_tau)
    h = load_library().lf_cache_create_ex(layers, batch, kv_heads, q_heads, head_dim, capacity,
                                          window, ctypes.byref(cfg))
    if not h:
        raise _create_failed()
    return h


def lf_cache_destroy(handle) -> int:
    return _check(load_library().lf_cache_destroy(handle))


def lf_prefill_fill(handle, layer, k, v, prompt_len: Sequence[int], max_prompt, stream=None) -> int:
    arr = (ctypes.c_int32 * len(prompt_len))(*[int(x) for x in prompt_len])
    return _check(load_library().lf_prefill_fill(handle, layer, _ptr(k), _ptr(v), arr,
                                                 int(max_prompt), _stream(stream)))


def lf_decode_step(handle, layer, q, k_new, v_new, out, evicted_slot, stream=None) -> int:
    return _check(load_library().lf_decode_step(handle, layer, _ptr(q), _ptr(k_new), _ptr(v_new),
                                                _ptr(out), _ptr(evicted_slot), _stream(stream)))


def lf_cache_check(handle, stream=None) -> int:
    """Return the device error bits (0 when clean); raise on a CUDA failure."""
    bits = ctypes.c_int32(0)
    code = load_library().lf_cache_check(handle, _stream(stream), ctypes.byref(bits))
    if code not in (LF_OK, LF_ERR_DEVICE):
        raise LFError(code, lf_last_error())
    return int(bits.value)


def lf_prefill_fill_noalloc(dst: LFLayout, layer, k, v, prompt_len: Sequence[int], max_prompt,
                            stream=None) -> int:
    arr = (ctypes.c_int32 * len(prompt_len))(*[int(x) for x in prompt_len])
    return _check(load_library().lf_prefill_fill_noalloc(ctypes.byref(dst), layer, _ptr(k), _ptr(v),
                                                         arr, int(max_prompt), _stream(stream)))


def lf_rkv_compress(handle, layer, q_obs, stream=None) -> int:
    return _check(load_library().lf_rkv_compress(handle, layer, _ptr(q_obs), _stream(stream)))


def lf_launch_plan(handle, layer):
    """The next step's plan of `layer`: None (whole units j, j + nc, ... per
    cluster), or (rounds, cuts) with cuts[j] = (unit, slot) where cluster j's
    range of the units past the whole rounds starts (cuts[nc] = (units, 0))."""
    lib = load_library()
    n = 256
    rounds = ctypes.c_int32(0)
    cu, cs = ((ctypes.c_int32 * n)() for _ in range(2))
    nc = lib.lf_launch_plan(handle, layer, ctypes.byref(rounds), cu, cs, n)
    if nc < 0:
        raise LFError(nc, lf_last_error())
    if nc == 0:
        return None
    return int(rounds.value), [(int(cu[j]), int(cs[j])) for j in range(nc + 1)]


def lf_launch_plan_for(occupancy: Sequence[int], cluster: int, clusters: int, max_items: int):
    """The planner on given per-unit occupancies: None or (rounds, cuts), as
    lf_launch_plan returns them."""
    lib = load_library()
    occ = (ctypes.c_int32 * len(occupancy))(*[int(x) for x in occupancy])
    rounds = ctypes.c_int32(0)
    cu, cs = ((ctypes.c_int32 * (clusters + 1))() for _ in range(2))
    nc = lib.lf_launch_plan_for(occ, len(occupancy), cluster, clusters, max_items,
                                ctypes.byref(rounds), cu, cs)
    if nc < 0:
        raise LFError(nc, lf_last_error())
    if nc == 0:
        return None
    return int(rounds.value), [(int(cu[j]), int(cs[j])) for j in range(nc + 1)]


def lf_cache_layout(handle) -> LFLayout:
    lay = LFLayout()
    _check(load_library().lf_cache_layout(handle, ctypes.byref(lay)))
    return lay


# ---- convenience owner ------------------------------------------------------

class _DevArray:
    """Minimal __cuda_array_interface__ exporter for a raw device pointer."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"data": (int(ptr), False), "shape": tuple(shape),
                                         "typestr": typestr, "version": 3, "strides": None}


def _view(ptr, shape, dtype: torch.dtype, device) -> torch.Tensor:
    typestr = {torch.float32: "<f4", torch.int32: "<i4", torch.int16: "<i2"}[dtype]
    return torch.as_tensor(_DevArray(ptr, shape, typestr), device=device)


class LFCache:
    """One LongFlow cache (owns the C handle).  Sizes as in ``lf_cache_create_ex``."""

    def __init__(self, layers, batch, kv_heads, q_heads, head_dim, capacity, window,
                 dtype="bf16", evict=True, budgets=None, cluster=0, stages=0, kernel="auto",
                 device=None, score="longflow", norm=1, sinks=0, deferred=False,
                 scope="kv_head", **rkv):
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        with torch.cuda.device(self.device):
            self.handle = lf_cache_create_ex(layers, batch, kv_heads, q_heads, head_dim, capacity,
                                             window, dtype, evict, budgets, cluster, stages,
                                             kernel, score, norm, sinks, deferred, scope, **rkv)
        self.layout = lf_cache_layout(self.handle)
        self.dtype = _TORCH_DTYPE[self.layout.dtype]
        self.layers, self.batch = layers, batch
        self.kv_heads, self.q_heads, self.head_dim = kv_heads, q_heads, head_dim
        self.capacity, self.window = capacity, window
        self.evict = self.layout.evict != LF_EVICT_OFF

    def close(self):
        if getattr(self, "handle", None):
            lf_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _expect(self, t, shape, name, dtype=None):
        dtype = dtype or self.dtype
        if not isinstance(t, torch.Tensor) or t.device != self.device or t.dtype != dtype \
                or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
            got = (tuple(t.shape), t.dtype, str(t.device)) if isinstance(t, torch.Tensor) else type(t)
            raise LFError(LF_ERR_ARG, f"{name}: expected contiguous {dtype} {tuple(shape)} on "
                                      f"{self.device}, got {got}")

    def prefill(self, layer, k, v, prompt_lens, stream=None):
        pmax = k.shape[2]
        self._expect(k, (self.batch, self.kv_heads, pmax, self.head_dim), "k")
        self._expect(v, (self.batch, self.kv_heads, pmax, self.head_dim), "v")
        lf_prefill_fill(self.handle, layer, k, v, list(prompt_lens), pmax, stream)

    def decode_step(self, layer, q, k_new, v_new, out=None, evicted=None, stream=None):
        b, hq, hkv, d = self.batch, self.q_heads, self.kv_heads, self.head_dim
        self._expect(q, (b, hq, d), "q")
        self._expect(k_new, (b, hkv, d), "k_new")
        self._expect(v_new, (b, hkv, d), "v_new")
        if out is None:
            out = torch.empty((b, hq, d), dtype=self.dtype, device=self.device)
        if evicted is None:
            evicted = torch.empty((b, hkv), dtype=torch.int32, device=self.device)
        self._expect(out, (b, hq, d), "out")
        self._expect(evicted, (b, hkv), "evicted", torch.int32)
        lf_decode_step(self.handle, layer, q, k_new, v_new, out, evicted, stream)
        return out, evicted

    def rkv_compress(self, layer, q_obs, stream=None):
        """R-KV compression of one layer; q_obs [batch][rkv_alpha][q_heads][head_dim]."""
        lay = self.layout
        self._expect(q_obs, (self.batch, lay.rkv_alpha, self.q_heads, self.head_dim), "q_obs")
        lf_rkv_compress(self.handle, layer, q_obs, stream)

    def plan(self, layer: int):
        """lf_launch_plan: None, or the (unit, slot) cuts of the next step of `layer`."""
        return lf_launch_plan(self.handle, layer)

    def check(self, stream=None) -> int:
        return lf_cache_check(self.handle, stream)

    def views(self):
        """Torch tensors aliasing the slab (no copy): k, v [L][b][H_kv][stride][d],
        vnorm, pos [L][b][H_kv][stride], count, next_pos [L][b][H_kv], budget [b];
        acc [L][b][H_kv][stride] (H2O) and pending [L][b][H_kv] (deferred), else None;
        split_cnt [split_units][2] (split launches), else None."""
        lay = self.layout
        L, b, g, s, d = lay.layers, lay.batch, lay.kv_heads, lay.slot_stride, lay.head_dim
        if self.dtype == torch.bfloat16:
            k = _view(lay.k, (L, b, g, s, d), torch.int16, self.device).view(torch.bfloat16)
            v = _view(lay.v, (L, b, g, s, d), torch.int16, self.device).view(torch.bfloat16)
        else:
            k = _view(lay.k, (L, b, g, s, d), torch.float32, self.device)
            v = _view(lay.v, (L, b, g, s, d), torch.float32, self.device)
        return {
            "k": k, "v": v,
            "vnorm": _view(lay.vnorm, (L, b, g, s), torch.float32, self.device),
            "pos": _view(lay.pos, (L, b, g, s), torch.int32, self.device),
            "count": _view(lay.count, (L, b, g), torch.int32, self.device),
            "next_pos": _view(lay.next_pos, (L, b, g), torch.int32, self.device),
            "budget": _view(lay.budget, (b,), torch.int32, self.device),
            "acc": (_view(lay.acc, (L, b, g, s), torch.float32, self.device)
                    if lay.acc else None),
            "pending": (_view(lay.pending, (L, b, g), torch.int32, self.device)
                        if lay.pending else None),
            "split_cnt": (_view(lay.split_cnt, (lay.split_units, 2), torch.int32, self.device)
                          if lay.split_cnt else None),
        }
