"""Python binding of libft (include/ft.h): argument marshalling only.

Every function here has the name of the C entry point it calls and passes
torch tensors as raw pointers.  All computation happens in libft's CUDA
kernels; there is no fallback: importing this package without a built
``libft.so`` raises, and a failing call raises ``FTError`` with the status.

Build the library with ``python -m expert_cache_streaming_fp32_b300.build``
(or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libft.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libft.so is not built ({LIB_PATH}); run python -m expert_cache_streaming_fp32_b300.build")

_lib = ctypes.CDLL(LIB_PATH)

# status / enums (values of include/ft.h)
FT_OK, FT_EINVAL, FT_ENOMEM, FT_ECUDA, FT_ETIMEOUT, FT_ESTATE, FT_EUNSUPPORTED, FT_EDEVICE, FT_EIO = range(9)
FT_INJECT_DEVICE_ALLOC, FT_INJECT_HOST_PIN, FT_INJECT_STREAM_EVENT = 1, 2, 3
FT_PLACE_GLOBAL_LRU, FT_PLACE_PREFILL_HOT, FT_PLACE_STATIC_SPLIT = 0, 1, 2
FT_FP4_BLOCK_SCALED, FT_FP4_EXPAND_BF16 = 0, 1
FT_W_F32, FT_W_BF16, FT_W_FP8E4M3, FT_W_NVFP4, FT_W_MXFP4 = range(5)
FT_X_F32, FT_X_BF16 = 0, 1

EXPORTED = [
    "ft_status_str", "ft_version", "ft_last_cuda_error", "ft_get_device_error", "ft_expert_layout_get",
    "ft_host_alloc", "ft_host_free", "ft_router_logits", "ft_route", "ft_permute", "ft_cache_create",
    "ft_cache_destroy", "ft_cache_n_waves", "ft_cache_step", "ft_cache_resize", "ft_cache_stats",
    "ft_cache_export", "ft_expert_grouped_workspace", "ft_expert_grouped", "ft_combine", "ft_stream_create",
    "ft_stream_layer", "ft_stream_layer_done", "ft_stream_bytes", "ft_stream_destroy", "ft_qsplit",
    "ft_expert_grouped_noalloc", "ft_debug_bounded_wait", "ft_cache_step_split", "ft_cache_fill_join",
    "ft_cache_set_fill_blocks", "ft_debug_inject_failure", "ft_debug_live_resources", "ft_pool_read",
    "ft_host_register", "ft_host_unregister", "ft_cache_reset", "ft_placement_replay", "ft_cpu_create",
    "ft_cpu_destroy", "ft_cpu_experts", "ft_cpu_experts_enqueue", "ft_cpu_status", "ft_route_fused",
    "ft_expert_set_fp4_path", "ft_debug_quant_fp4", "ft_debug_host_simd",
]
FT_NOALLOC_MAX_ELEMS = 1 << 20
FT_TC_WIDE_ASSIGNMENTS = 2048
FT_CC_MAX_ASSIGNMENTS = 8
FT_ROUTE_ARRIVAL_WORDS = 16


class FTError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _lib.ft_status_str(status).decode()
        if status == FT_ECUDA:
            msg += f" (cudaError {_lib.ft_last_cuda_error()})"
        super().__init__(f"{fn}: {msg} [{status}]")
        self.status = status


class ExpertLayout(ctypes.Structure):
    _fields_ = [("bytes", ctypes.c_uint64), ("payload_bytes", ctypes.c_uint64), ("off_val", ctypes.c_uint64 * 3),
                ("off_scale", ctypes.c_uint64 * 3), ("off_gscale", ctypes.c_uint64)]


class CacheConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("n_experts", ctypes.c_int), ("n_phys_layers", ctypes.c_int),
                ("n_slots", ctypes.c_int), ("max_slots", ctypes.c_int), ("slot_bytes", ctypes.c_uint64),
                ("host_pool", ctypes.c_void_p), ("slot_pool", ctypes.c_void_p)]


class CacheStats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("fills", ctypes.c_uint64),
                ("externals", ctypes.c_uint64), ("bytes_h2d", ctypes.c_uint64)]


class CpuJob(ctypes.Structure):
    _fields_ = [("host_pool", ctypes.c_void_p), ("slot_bytes", ctypes.c_uint64), ("wtype", ctypes.c_int),
                ("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("phys_layer", ctypes.c_int), ("x", ctypes.c_void_p), ("x_type", ctypes.c_int), ("T", ctypes.c_int),
                ("k", ctypes.c_int), ("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("ext_flags", ctypes.c_void_p), ("partial", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_sigs = {
    "ft_status_str": (ctypes.c_char_p, [_I]),
    "ft_version": (_I, []),
    "ft_last_cuda_error": (_I, []),
    "ft_get_device_error": (_I, [ctypes.POINTER(_I)]),
    "ft_expert_layout_get": (_I, [_I, _I, _I, ctypes.POINTER(ExpertLayout)]),
    "ft_host_alloc": (_I, [ctypes.c_uint64, ctypes.POINTER(_P)]),
    "ft_host_free": (_I, [_P]),
    "ft_router_logits": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _P]),
    "ft_route": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "ft_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "ft_expert_set_fp4_path": (_I, [_I]),
    "ft_debug_quant_fp4": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "ft_route_fused": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ft_cache_create": (_I, [ctypes.POINTER(CacheConfig), ctypes.POINTER(_P)]),
    "ft_cache_destroy": (_I, [_P]),
    "ft_cache_n_waves": (_I, [_P]),
    "ft_cache_step": (_I, [_P, _I, _P, ctypes.c_double, _I, _P, _P, _P, _P]),
    "ft_cache_step_split": (_I, [_P, _I, _P, ctypes.c_double, _I, _P, _P, _P, _P, _P, _P]),
    "ft_cache_fill_join": (_I, [_P, _P]),
    "ft_cache_set_fill_blocks": (_I, [_P, _I]),
    "ft_cache_resize": (_I, [_P, _I]),
    "ft_cache_reset": (_I, [_P]),
    "ft_cpu_create": (_I, [_I, ctypes.POINTER(_P)]),
    "ft_cpu_destroy": (_I, [_P]),
    "ft_cpu_experts": (_I, [_P, ctypes.POINTER(CpuJob)]),
    "ft_cpu_experts_enqueue": (_I, [_P, ctypes.POINTER(CpuJob), _P]),
    "ft_cpu_status": (_I, [_P]),
    "ft_placement_replay": (_I, [_I, _I, _I, _I, _P, _P, _I, _I, ctypes.POINTER(ctypes.c_uint64),
                                 ctypes.POINTER(ctypes.c_uint64)]),
    "ft_cache_stats": (_I, [_P, ctypes.POINTER(CacheStats)]),
    "ft_cache_export": (_I, [_P, _P, _P, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_uint32)]),
    "ft_expert_grouped_workspace": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "ft_expert_grouped": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, ctypes.c_uint64, _I, _P, _P,
                               ctypes.c_size_t, _P]),
    "ft_combine": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "ft_stream_create": (_I, [_P, _I, ctypes.POINTER(_P)]),
    "ft_stream_layer": (_I, [_P, _I, _I, _P, _P]),
    "ft_stream_layer_done": (_I, [_P, _I, _P]),
    "ft_stream_bytes": (_I, [_P, ctypes.POINTER(ctypes.c_uint64)]),
    "ft_stream_destroy": (_I, [_P]),
    "ft_qsplit": (_I, [_I, ctypes.c_double, ctypes.c_double]),
    "ft_expert_grouped_noalloc": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, ctypes.c_uint64, _I, _P, _P]),
    "ft_debug_bounded_wait": (_I, [ctypes.c_int64, _P, _P]),
    "ft_debug_inject_failure": (_I, [_I, _I]),
    "ft_debug_live_resources": (_I, [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "ft_debug_host_simd": (_I, [_I]),
    "ft_pool_read": (_I, [ctypes.c_char_p, ctypes.c_uint64, _P, ctypes.c_uint64, _I]),
    "ft_host_register": (_I, [_P, ctypes.c_uint64]),
    "ft_host_unregister": (_I, [_P]),
}
for _name, (_res, _args) in _sigs.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def _check(fn: str, status: int):
    if status != FT_OK:
        raise FTError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(s):
    if s is None:
        s = torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _xtype(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return FT_X_BF16
    if x.dtype == torch.float32:
        return FT_X_F32
    raise TypeError(f"activations must be bf16 or fp32, got {x.dtype}")


def lib():
    return _lib


# ---------------------------------------------------------------- thin wrappers

def ft_version() -> int:
    return _lib.ft_version()


def ft_status_str(status: int) -> str:
    return _lib.ft_status_str(status).decode()


def ft_get_device_error() -> int:
    code = _I(0)
    st = _lib.ft_get_device_error(ctypes.byref(code))
    if st not in (FT_OK, FT_EDEVICE):
        _check("ft_get_device_error", st)
    return code.value


def ft_expert_layout_get(wtype: int, hidden: int, inter: int) -> ExpertLayout:
    L = ExpertLayout()
    _check("ft_expert_layout_get", _lib.ft_expert_layout_get(wtype, hidden, inter, ctypes.byref(L)))
    return L


def ft_debug_bounded_wait(limit_ns: int, completed, stream=None):
    """Runs the bounded-wait failure path on purpose (a barrier that nothing completes)."""
    _check("ft_debug_bounded_wait", _lib.ft_debug_bounded_wait(int(limit_ns), _ptr(completed), _stream(stream)))


def ft_debug_inject_failure(site: int, after: int):
    """Arms (after >= 0) or disarms (after < 0) a host-side failure at one site of the library."""
    _check("ft_debug_inject_failure", _lib.ft_debug_inject_failure(site, after))


def ft_debug_live_resources():
    """(device allocations, streams + events) held by the library's handles."""
    a, b = ctypes.c_int64(0), ctypes.c_int64(0)
    _check("ft_debug_live_resources", _lib.ft_debug_live_resources(ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


HOST_FORMS = ("portable", "avx2", "avx512")


def ft_debug_host_simd(mode: int = -1) -> int:
    """Selects the host executor's row form (0 portable, 1 AVX2, 2 AVX-512; each where the CPU
    runs it, else the best below it), or only asks (-1); returns the form in use before."""
    return _lib.ft_debug_host_simd(mode)


def ft_pool_read(path: str, offset: int, dst_ptr: int, nbytes: int, threads: int = 0):
    _check("ft_pool_read", _lib.ft_pool_read(os.fsencode(path), offset, ctypes.c_void_p(dst_ptr), nbytes, threads))


def ft_host_register(ptr: int, nbytes: int):
    _check("ft_host_register", _lib.ft_host_register(ctypes.c_void_p(ptr), nbytes))


def ft_host_unregister(ptr: int):
    _check("ft_host_unregister", _lib.ft_host_unregister(ctypes.c_void_p(ptr)))


def ft_placement_replay(policy: int, n_layers: int, n_experts: int, capacity: int, trace, prefill_counts=None):
    """(accesses, misses) of a routing trace (int32 array [steps, layers, width]) under a placement policy."""
    import numpy as np
    tr = np.ascontiguousarray(trace, dtype=np.int32)
    assert tr.ndim == 3 and tr.shape[1] == n_layers
    pc = None if prefill_counts is None else np.ascontiguousarray(prefill_counts, dtype=np.int32).reshape(-1)
    acc, miss = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check("ft_placement_replay", _lib.ft_placement_replay(
        policy, n_layers, n_experts, capacity, None if pc is None else pc.ctypes.data_as(_P), tr.ctypes.data_as(_P),
        tr.shape[0], tr.shape[2], ctypes.byref(acc), ctypes.byref(miss)))
    return acc.value, miss.value


def ft_qsplit(m: int, bw_fill: float, bw_host: float) -> int:
    return _lib.ft_qsplit(m, bw_fill, bw_host)


def ft_router_logits(x, w_router, bias, logits, stream=None):
    T, H = x.shape
    E = w_router.shape[0]
    _check("ft_router_logits", _lib.ft_router_logits(_ptr(x), _xtype(x), _ptr(w_router), _ptr(bias), T, H, E,
                                                     _ptr(logits), _stream(stream)))


def ft_route(logits, k, topk_idx, topk_w, stream=None):
    T, E = logits.shape
    _check("ft_route", _lib.ft_route(_ptr(logits), T, E, k, _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


def ft_permute(topk_idx, E, counts, offsets, perm, inv, stream=None):
    T, k = topk_idx.shape
    _check("ft_permute", _lib.ft_permute(_ptr(topk_idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm),
                                         _ptr(inv), _stream(stream)))


def ft_route_fused(x, w_router, bias, k, logits, topk_idx, topk_w, counts, offsets, perm, inv, arrivals,
                   stream=None):
    """``arrivals``: a zeroed device int32/uint32 tensor of FT_ROUTE_ARRIVAL_WORDS words, one per
    routing that may be in flight at a time; every call leaves it zero."""
    T, H = x.shape
    E = w_router.shape[0]
    if arrivals is not None and arrivals.numel() < FT_ROUTE_ARRIVAL_WORDS:
        raise ValueError("arrivals needs FT_ROUTE_ARRIVAL_WORDS words")
    _check("ft_route_fused", _lib.ft_route_fused(
        _ptr(x), _xtype(x), _ptr(w_router), _ptr(bias), T, H, E, k, _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
        _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(arrivals), _stream(stream)))


def ft_expert_set_fp4_path(path: int):
    """FT_FP4_BLOCK_SCALED (block-scaled FP4 MMA, FP4 activations) or FT_FP4_EXPAND_BF16 (exact expansion)."""
    _check("ft_expert_set_fp4_path", _lib.ft_expert_set_fp4_path(path))


def ft_debug_quant_fp4(x, wtype, q, scales, stream=None):
    rows, K = x.shape
    _check("ft_debug_quant_fp4", _lib.ft_debug_quant_fp4(_ptr(x), _xtype(x), rows, K, wtype, _ptr(q), _ptr(scales),
                                                         _stream(stream)))


def ft_expert_grouped_workspace(T, k, hidden, inter) -> int:
    return _lib.ft_expert_grouped_workspace(T, k, hidden, inter)


def ft_expert_grouped(x, k, inter, E, wtype, perm, offsets, slot_of, slot_pool, slot_bytes, pool_slots, y,
                      workspace, stream=None):
    T, H = x.shape
    _check("ft_expert_grouped", _lib.ft_expert_grouped(
        _ptr(x), _xtype(x), T, k, H, inter, E, wtype, _ptr(perm), _ptr(offsets), _ptr(slot_of), _ptr(slot_pool),
        slot_bytes, pool_slots, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def ft_expert_grouped_noalloc(x, k, inter, E, wtype, perm, offsets, slot_of, slot_pool, slot_bytes, pool_slots, y,
                              stream=None):
    """ft_expert_grouped without a workspace, for callers that cannot allocate device memory.

    The intermediate uses a fixed 4 MiB array inside libft (T*k*inter must not
    exceed FT_NOALLOC_MAX_ELEMS); calls that overlap on the GPU race on it.
    """
    T, H = x.shape
    _check("ft_expert_grouped_noalloc", _lib.ft_expert_grouped_noalloc(
        _ptr(x), _xtype(x), T, k, H, inter, E, wtype, _ptr(perm), _ptr(offsets), _ptr(slot_of), _ptr(slot_pool),
        slot_bytes, pool_slots, _ptr(y), _stream(stream)))


def ft_combine(y, inv, topk_idx, topk_w, ext_flags, ext_partial, E, out, stream=None):
    T, k = topk_idx.shape
    H = out.shape[1]
    _check("ft_combine", _lib.ft_combine(_ptr(y), _ptr(inv), _ptr(topk_idx), _ptr(topk_w), _ptr(ext_flags),
                                         _ptr(ext_partial), T, k, H, E, _ptr(out), _stream(stream)))


# ---------------------------------------------------------------- pinned pool

class PinnedBuffer:
    """Pinned, device-mapped host memory from ft_host_alloc, viewed as a uint8 tensor."""

    def __init__(self, nbytes: int):
        p = _P()
        _check("ft_host_alloc", _lib.ft_host_alloc(nbytes, ctypes.byref(p)))
        self.ptr = p.value
        self.nbytes = nbytes
        arr = (ctypes.c_uint8 * nbytes).from_address(self.ptr)
        import numpy as np
        self.tensor = torch.from_numpy(np.ctypeslib.as_array(arr))

    def free(self):
        if self.ptr:
            self.tensor = None
            _check("ft_host_free", _lib.ft_host_free(ctypes.c_void_p(self.ptr)))
            self.ptr = 0

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class RegisteredBuffer:
    """Read-then-pin host memory: a page-aligned anonymous mapping that is filled
    first (its pages are faulted in by that write) and pinned afterwards with
    ft_host_register, viewed as a uint8 tensor.  ``pin()`` must come before the
    GPU reads it."""

    def __init__(self, nbytes: int):
        import mmap
        import numpy as np
        self.map = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        arr = np.frombuffer(self.map, dtype=np.uint8)
        self.ptr = arr.ctypes.data
        self.nbytes = nbytes
        self.tensor = torch.from_numpy(arr)
        self.pinned = False

    def read(self, path: str, offset: int = 0, threads: int = 0):
        """Fills the whole buffer from a pool file with libft's parallel reader."""
        ft_pool_read(path, offset, self.ptr, self.nbytes, threads)

    def pin(self):
        if not self.pinned:
            ft_host_register(self.ptr, self.nbytes)
            self.pinned = True

    def free(self):
        if self.ptr:
            if self.pinned:
                ft_host_unregister(self.ptr)
                self.pinned = False
            self.tensor = None
            self.ptr = 0
            try:
                self.map.close()
            except BufferError:       # a view is still alive; the mapping goes with it
                pass

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


# ---------------------------------------------------------------- cache

class Cache:
    """Owner of an ft_cache handle (the tables live in libft; the pools are the caller's)."""

    def __init__(self, n_layers, n_experts, n_phys_layers, n_slots, max_slots, slot_bytes, host_pool_ptr,
                 slot_pool: torch.Tensor):
        cfg = CacheConfig(n_layers, n_experts, n_phys_layers, n_slots, max_slots, slot_bytes, host_pool_ptr,
                          slot_pool.data_ptr())
        h = _P()
        _check("ft_cache_create", _lib.ft_cache_create(ctypes.byref(cfg), ctypes.byref(h)))
        self.h = h
        self.E, self.max_slots, self.slot_pool = n_experts, max_slots, slot_pool

    def destroy(self):
        if self.h:
            _lib.ft_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def n_waves(self) -> int:
        return _lib.ft_cache_n_waves(self.h)

    def step(self, layer, counts, fill_ratio, wave, slot_of, ext_flags=None, step_counts=None, stream=None):
        _check("ft_cache_step", _lib.ft_cache_step(self.h, layer, _ptr(counts), float(fill_ratio), wave,
                                                   _ptr(slot_of), _ptr(ext_flags), _ptr(step_counts),
                                                   _stream(stream)))

    def step_split(self, layer, counts, fill_ratio, wave, slot_hit, slot_fill, ext_flags=None, step_counts=None,
                   stream=None, fill_stream=None):
        _check("ft_cache_step_split",
               _lib.ft_cache_step_split(self.h, layer, _ptr(counts), float(fill_ratio), wave, _ptr(slot_hit),
                                        _ptr(slot_fill), _ptr(ext_flags), _ptr(step_counts), _stream(stream),
                                        _stream(fill_stream)))

    def set_fill_blocks(self, blocks: int):
        _check("ft_cache_set_fill_blocks", _lib.ft_cache_set_fill_blocks(self.h, blocks))

    def fill_join(self, stream=None):
        _check("ft_cache_fill_join", _lib.ft_cache_fill_join(self.h, _stream(stream)))

    def resize(self, n_slots):
        _check("ft_cache_resize", _lib.ft_cache_resize(self.h, n_slots))

    def reset(self):
        """Cold restart: every slot empty, clock and counters zero (graphs over the handle stay valid)."""
        _check("ft_cache_reset", _lib.ft_cache_reset(self.h))

    def stats(self) -> CacheStats:
        s = CacheStats()
        _check("ft_cache_stats", _lib.ft_cache_stats(self.h, ctypes.byref(s)))
        return s

    def export(self):
        import numpy as np
        key = np.zeros(self.max_slots, dtype=np.int32)
        stamp = np.zeros(self.max_slots, dtype=np.uint32)
        n = _I(0)
        clk = ctypes.c_uint32(0)
        _check("ft_cache_export", _lib.ft_cache_export(self.h, key.ctypes.data_as(_P), stamp.ctypes.data_as(_P),
                                                       ctypes.byref(n), ctypes.byref(clk)))
        return key[: n.value].copy(), stamp[: n.value].copy(), clk.value


class CpuExperts:
    """Owner of an ft_cpu handle: the host-side expert executor (a pool of CPU threads)."""

    def __init__(self, threads: int = 0):
        h = _P()
        _check("ft_cpu_create", _lib.ft_cpu_create(threads, ctypes.byref(h)))
        self.h = h
        self._enqueued = []

    @staticmethod
    def job(host_pool_ptr, slot_bytes, wtype, hidden, inter, n_experts, phys_layer, x, T, k, topk_idx, topk_w,
            ext_flags, partial) -> CpuJob:
        """A job over host tensors (x [T, H] bf16/fp32, topk_idx/topk_w [T, k], ext_flags [E], partial [T, H] fp32)."""
        for t in (x, topk_idx, topk_w, ext_flags, partial):
            assert not t.is_cuda and t.is_contiguous()
        job = CpuJob(host_pool_ptr, slot_bytes, wtype, hidden, inter, n_experts, phys_layer, x.data_ptr(), _xtype(x),
                     T, k, topk_idx.data_ptr(), topk_w.data_ptr(), ext_flags.data_ptr(), partial.data_ptr())
        job._tensors = (x, topk_idx, topk_w, ext_flags, partial)   # the job's pointers stay valid while it lives
        return job

    def run(self, job: CpuJob):
        _check("ft_cpu_experts", _lib.ft_cpu_experts(self.h, ctypes.byref(job)))

    def enqueue(self, job: CpuJob, stream=None):
        """The handle keeps the job (and runs it at every replay of a captured stream), so the
        job and its tensors are kept here until destroy."""
        _check("ft_cpu_experts_enqueue", _lib.ft_cpu_experts_enqueue(self.h, ctypes.byref(job), _stream(stream)))
        self._enqueued.append(job)

    def status(self) -> int:
        return _lib.ft_cpu_status(self.h)

    def destroy(self):
        if self.h:
            _lib.ft_cpu_destroy(self.h)
            self.h = None
            self._enqueued = []

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class Stream:
    """Owner of an ft_stream handle (whole-layer double-buffered prefill)."""

    def __init__(self, cache: Cache, serialized: bool = False):
        h = _P()
        _check("ft_stream_create", _lib.ft_stream_create(cache.h, 1 if serialized else 0, ctypes.byref(h)))
        self.h = h
        self.cache = cache            # the stream handle points into the cache handle

    def layer(self, layer, next_layer, slot_of, stream=None):
        _check("ft_stream_layer", _lib.ft_stream_layer(self.h, layer, next_layer, _ptr(slot_of), _stream(stream)))

    def layer_done(self, layer, stream=None):
        _check("ft_stream_layer_done", _lib.ft_stream_layer_done(self.h, layer, _stream(stream)))

    def bytes(self) -> int:
        b = ctypes.c_uint64(0)
        _check("ft_stream_bytes", _lib.ft_stream_bytes(self.h, ctypes.byref(b)))
        return b.value

    def destroy(self):
        if self.h:
            st = _lib.ft_stream_destroy(self.h)
            self.h = None
            _check("ft_stream_destroy", st)


from .layer import (SPLIT_MAX_ASSIGNMENTS, SPLIT_MIN_ASSIGNMENTS, ExpertPool, HostBranch, MoELayer,  # noqa: E402,F401
                    pack_expert, split_pays)
