"""Python binding of libnsmuon.so, the GB300 owner-side Muon optimizer step.

This module only marshals arguments: it turns torch tensors into device pointers and
host tables into C arrays and calls the C ABI declared in ``include/nsmuon.h``.  Every
step of the optimizer runs in the library's CUDA kernels; there is no CPU fallback, and
importing the binding fails loudly when the library has not been built.

Names follow the pages ("DeepSpeed 集成 Muon 优化器实战"): ``ns_method`` is
``"standard"`` or ``"gram"`` (default ``"gram"``), ``muon_lr`` / ``adam_lr`` override a
group's ``lr``, the Muon group defaults are lr 0.02 and momentum 0.95, and the Adam group
defaults are lr 3e-4, betas (0.9, 0.95) and eps 1e-10.
"""

from __future__ import annotations

import ctypes
import os
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_REGULAR = os.path.join(_HERE, "libnsmuon.so")
# the bounds-checked build: every kernel tests each access to a matrix's elements before
# making it, records a failure (NSM_ERR_BOUNDS) and skips the access
LIB_CHECKED = os.path.join(_HERE, "libnsmuon_checked.so")
# NSM_CHECKED=1 in the environment makes this process load the checked build
LIB_PATH = LIB_CHECKED if os.environ.get("NSM_CHECKED") == "1" else LIB_REGULAR

NSM_OK = 0
NSM_ERR_NULL = -1
NSM_ERR_SHAPE = -2
NSM_ERR_OFFSET = -3
NSM_ERR_ALIGN = -4
NSM_ERR_METHOD = -5
NSM_ERR_WORKSPACE = -6
NSM_ERR_CUDA = -7
NSM_ERR_TIMEOUT = -8
NSM_ERR_ARG = -9
NSM_ERR_BOUNDS = -10

NS_METHODS = {"standard": 0, "gram": 1, "standard_bf16": 2}
NS_METHOD_DEFAULT = "gram"
NS_STEPS_DEFAULT = 5
MUON_LR_DEFAULT = 0.02
MUON_MOMENTUM_DEFAULT = 0.95
ADAM_LR_DEFAULT = 3e-4
ADAM_BETAS_DEFAULT = (0.9, 0.95)
ADAM_EPS_DEFAULT = 1e-10

_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_i64p = ctypes.POINTER(ctypes.c_int64)
_vp = ctypes.c_void_p

_lib: Optional[ctypes.CDLL] = None


class NsmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"nsmuon error {code}: {message}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Loads libnsmuon.so, or libnsmuon_checked.so when NSM_CHECKED=1 (both built in-tree
    by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
    L = ctypes.CDLL(LIB_PATH)
    L.nsm_version.restype = ctypes.c_int
    L.nsm_last_error.restype = ctypes.c_char_p
    L.nsm_last_launch_count.restype = ctypes.c_int
    L.nsm_route.argtypes = [ctypes.c_char_p, ctypes.c_int]
    L.nsm_route.restype = ctypes.c_int
    L.nsm_pack.argtypes = [_c_i32p, ctypes.c_int, ctypes.c_int64, _c_i64p, _c_i64p]
    L.nsm_pack.restype = ctypes.c_int
    _c_ip = ctypes.POINTER(ctypes.c_int)
    L.nsm_input_exponent.argtypes = [ctypes.c_float, ctypes.c_int, ctypes.c_int, _c_ip, _c_ip, _c_ip]
    L.nsm_input_exponent.restype = ctypes.c_int
    L.nsm_assign_owners.argtypes = [_c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, _c_i32p, _c_i64p]
    L.nsm_assign_owners.restype = ctypes.c_int
    L.nsm_workspace_iterate.argtypes = [_c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.POINTER(ctypes.c_size_t),
                                        ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    L.nsm_workspace_iterate.restype = ctypes.c_int
    L.muon_workspace_bytes.argtypes = [_c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.muon_workspace_bytes.restype = ctypes.c_size_t
    L.muon_step.argtypes = [_vp, _vp, _vp, _c_i64p, _c_i32p, ctypes.c_int, ctypes.c_float,
                            ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, _vp, ctypes.c_size_t, _vp]
    L.muon_step.restype = ctypes.c_int
    L.muon_step_with_copy.argtypes = [_vp, _vp, _vp, _vp, _c_i64p, _c_i32p, ctypes.c_int,
                                      ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
    L.muon_step_with_copy.restype = ctypes.c_int
    L.muon_orthogonalize.argtypes = [_vp, _vp, _c_i64p, _c_i32p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _vp, ctypes.c_size_t, _vp]
    L.muon_orthogonalize.restype = ctypes.c_int
    L.muon_orthogonalize_noalloc.argtypes = [_vp, _vp, _c_i64p, _c_i32p, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, _vp]
    L.muon_orthogonalize_noalloc.restype = ctypes.c_int
    L.adamw_step.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                             ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int, _vp]
    L.adamw_step.restype = ctypes.c_int
    L.nsm_gemm.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp,
                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                           ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                           ctypes.c_float, _vp, ctypes.c_size_t, _vp]
    L.nsm_gemm.restype = ctypes.c_int
    L.nsm_gemm_scratch_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.nsm_gemm_scratch_bytes.restype = ctypes.c_size_t
    L.nsm_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int)]
    L.nsm_device_status.restype = ctypes.c_int
    _ip = ctypes.POINTER(ctypes.c_int)
    L.nsm_device_status_detail.argtypes = [_vp, _ip, _ip, _ip, _ip]
    L.nsm_device_status_detail.restype = ctypes.c_int
    L.nsm_set_option.argtypes = [ctypes.c_int, ctypes.c_int]
    L.nsm_set_option.restype = ctypes.c_int
    L.nsm_get_option.argtypes = [ctypes.c_int]
    L.nsm_get_option.restype = ctypes.c_int
    L.nsm_status_selftest.argtypes = [ctypes.c_int, _vp]
    L.nsm_status_selftest.restype = ctypes.c_int
    L.nsm_bounds_selftest.argtypes = [_vp]
    L.nsm_bounds_selftest.restype = ctypes.c_int
    L.nsm_copy_to_device.argtypes = [_vp, _vp, ctypes.c_size_t, ctypes.c_int, _vp]
    L.nsm_copy_to_device.restype = ctypes.c_int
    L.nsm_timing_enable.argtypes = [ctypes.c_int]
    L.nsm_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), _c_i64p,
                                  ctypes.POINTER(ctypes.c_double)]
    L.nsm_timing_read_kind.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double), _c_i64p,
                                       ctypes.POINTER(ctypes.c_double)]
    _lib = L
    return L


def _check(rc: int) -> int:
    if rc < 0:
        raise NsmError(rc, last_error())
    return rc


def last_error() -> str:
    return lib().nsm_last_error().decode("utf-8", "replace")


def version() -> int:
    return lib().nsm_version()


def last_launch_count() -> int:
    return lib().nsm_last_launch_count()


def route(name: str, ndim: int) -> bool:
    """Muon (True) or AdamW (False) for a named parameter of ``ndim`` dimensions."""
    return bool(_check(lib().nsm_route(name.encode("utf-8"), int(ndim))))


def input_exponent(max_abs: float, hint=None) -> Tuple[int, int, bool]:
    """(k, next hint, store again) of the stored input's exponent rule for a matrix whose
    largest |U| is ``max_abs`` (a float32 value), with the step's hint or without one."""
    k, nxt, store = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().nsm_input_exponent(float(max_abs), 0 if hint is None else 1, 0 if hint is None else int(hint),
                                    ctypes.byref(k), ctypes.byref(nxt), ctypes.byref(store)))
    return k.value, nxt.value, bool(store.value)


def _shapes_array(shapes: Sequence[Tuple[int, int]]) -> np.ndarray:
    arr = np.ascontiguousarray(np.asarray(shapes, dtype=np.int32).reshape(-1, 2))
    return arr


def _i32p(a: np.ndarray):
    return a.ctypes.data_as(_c_i32p)


def _i64p(a: np.ndarray):
    return a.ctypes.data_as(_c_i64p)


def pack(shapes: Sequence[Tuple[int, int]], align: int = 64) -> Tuple[np.ndarray, int]:
    """Offsets (int64 elements) and total length of the packed buffer for ``shapes``."""
    s = _shapes_array(shapes)
    n = s.shape[0]
    offs = np.zeros(n, dtype=np.int64)
    total = np.zeros(1, dtype=np.int64)
    _check(lib().nsm_pack(_i32p(s), n, int(align), _i64p(offs), _i64p(total)))
    return offs, int(total[0])


def assign_owners(shapes: Sequence[Tuple[int, int]], world: int, ns_method=NS_METHOD_DEFAULT,
                  ns_steps: int = NS_STEPS_DEFAULT) -> Tuple[np.ndarray, np.ndarray]:
    """Owner rank of every matrix (LPT on Newton-Schulz flops) and the flops per owner."""
    s = _shapes_array(shapes)
    owner = np.zeros(s.shape[0], dtype=np.int32)
    load = np.zeros(int(world), dtype=np.int64)
    _check(lib().nsm_assign_owners(_i32p(s), s.shape[0], int(world), method_code(ns_method),
                                   int(ns_steps), _i32p(owner), _i64p(load)))
    return owner, load


def owner_table(shapes: Sequence[Tuple[int, int]], owner: Sequence[int], rank: int,
                align: int = 64):
    """The packed table of one owner: (indices of its matrices, their shapes, offsets in its
    own packed buffer, that buffer's length)."""
    idx = [i for i, o in enumerate(owner) if int(o) == int(rank)]
    sub = [tuple(shapes[i]) for i in idx]
    if not sub:
        return idx, sub, np.zeros(0, dtype=np.int64), 0
    offs, total = pack(sub, align)
    return idx, sub, offs, total


# "Z2 与 Z3 模式" §每步通信字节数 and §显存开销: communication per step on a shard group of
# N ranks, in elements of the Muon-target parameters P_M, and the steady-state memory of
# the packed buffers.
DMUON_COMM_FACTORS = {"naive_z2": 3, "dmuon_z2": 2, "naive_z3": 4, "dmuon_z3": 3}


def dmuon_comm_elements(mode: str, world: int, p_m: float) -> float:
    """Elements each step moves on the shard group: k (N-1)/N P_M (k per mode)."""
    return DMUON_COMM_FACTORS[mode] * (world - 1) / world * p_m


def dmuon_packed_memory_elements(mode: str, world: int, p_m: float,
                                 max_layer_p_m: float = 0.0) -> float:
    """Steady-state elements of owned packed buffers per rank: P_M / N under Z2 (all
    resident), one layer's buffer (max_layer_P_M) under Z3."""
    if mode == "dmuon_z2":
        return p_m / world
    if mode == "dmuon_z3":
        return max_layer_p_m
    raise ValueError(mode)


def method_code(ns_method) -> int:
    if isinstance(ns_method, str):
        if ns_method not in NS_METHODS:
            raise ValueError(f"ns_method must be one of {sorted(NS_METHODS)}")
        return NS_METHODS[ns_method]
    return int(ns_method)


def workspace_bytes(shapes: Sequence[Tuple[int, int]], ns_method=NS_METHOD_DEFAULT,
                    ns_steps: int = NS_STEPS_DEFAULT) -> int:
    s = _shapes_array(shapes)
    b = lib().muon_workspace_bytes(_i32p(s), s.shape[0], method_code(ns_method), int(ns_steps))
    if b == 0:
        raise NsmError(NSM_ERR_ARG, last_error())
    return int(b)


def workspace_iterate(shapes: Sequence[Tuple[int, int]], i: int, buf: int, ns_method=NS_METHOD_DEFAULT,
                      ns_steps: int = NS_STEPS_DEFAULT) -> Tuple[int, int, int]:
    """(byte offset, m, row stride) of matrix i's m x m buffer `buf` in the workspace;
    m = 0 when its chain runs in the small-matrix kernel."""
    s = _shapes_array(shapes)
    off = ctypes.c_size_t(0)
    m = ctypes.c_int(0)
    ld = ctypes.c_int(0)
    _check(lib().nsm_workspace_iterate(_i32p(s), s.shape[0], method_code(ns_method), int(ns_steps), int(i),
                                       int(buf), ctypes.byref(off), ctypes.byref(m), ctypes.byref(ld)))
    return off.value, m.value, ld.value


def mm_buffers(ns_method=NS_METHOD_DEFAULT) -> int:
    """Number of m x m workspace buffers of a method (2 standard forms, 4 gram)."""
    return 4 if method_code(ns_method) == NS_METHODS["gram"] else 2


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream_ptr(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def muon_step(grads, params, momentum, offsets, shapes, lr: float = MUON_LR_DEFAULT,
              wd: float = 0.0, mu: float = MUON_MOMENTUM_DEFAULT,
              ns_method=NS_METHOD_DEFAULT, ns_steps: int = NS_STEPS_DEFAULT,
              nesterov: bool = True, workspace=None, stream=None, params_bf16=None) -> None:
    """One owner-side Muon step on packed buffers (bf16 grads, fp32 params/momentum).

    With ``params_bf16`` (a bf16 buffer of the same length) the step also writes the bf16
    copy of the updated parameters, the buffer an owner broadcasts."""
    s = _shapes_array(shapes)
    o = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    ws_size = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().muon_step_with_copy(_ptr(grads), _ptr(params), _ptr(momentum), _ptr(params_bf16),
                                     _i64p(o), _i32p(s), s.shape[0], float(lr), float(wd), float(mu),
                                     method_code(ns_method), int(ns_steps), 1 if nesterov else 0,
                                     _ptr(workspace), ws_size, _stream_ptr(stream)))


def muon_orthogonalize(inp, out, offsets, shapes, ns_method=NS_METHOD_DEFAULT,
                       ns_steps: int = NS_STEPS_DEFAULT, workspace=None, stream=None) -> None:
    """Newton-Schulz orthogonalisation of every matrix of a packed bf16 buffer."""
    s = _shapes_array(shapes)
    o = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    ws_size = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().muon_orthogonalize(_ptr(inp), _ptr(out), _i64p(o), _i32p(s), s.shape[0],
                                    method_code(ns_method), int(ns_steps), _ptr(workspace),
                                    ws_size, _stream_ptr(stream)))


def muon_orthogonalize_noalloc(inp, out, offsets, shapes, ns_method=NS_METHOD_DEFAULT,
                               ns_steps: int = NS_STEPS_DEFAULT, stream=None) -> None:
    """muon_orthogonalize without a workspace, for callers that cannot allocate device
    memory (a framework pool that owns all of it, a loop that cannot take an allocation's
    synchronisation).  Uses a 64 MiB array of device memory the library itself holds;
    tables that do not fit raise NsmError(NSM_ERR_WORKSPACE).  Calls that overlap on the
    GPU race on that array: keep them on one stream."""
    s = _shapes_array(shapes)
    o = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    _check(lib().muon_orthogonalize_noalloc(_ptr(inp), _ptr(out), _i64p(o), _i32p(s), s.shape[0],
                                            method_code(ns_method), int(ns_steps),
                                            _stream_ptr(stream)))


def adamw_step(grads, params, exp_avg, exp_avg_sq, lr: float = ADAM_LR_DEFAULT,
               beta1: float = ADAM_BETAS_DEFAULT[0], beta2: float = ADAM_BETAS_DEFAULT[1],
               eps: float = ADAM_EPS_DEFAULT, wd: float = 0.0, step: int = 1,
               stream=None) -> None:
    """Fused AdamW on one flat group (bf16 grads, fp32 params and moments)."""
    numel = 0 if params is None else params.numel()
    _check(lib().adamw_step(_ptr(grads), _ptr(params), _ptr(exp_avg), _ptr(exp_avg_sq), numel,
                            float(lr), float(beta1), float(beta2), float(eps), float(wd),
                            int(step), _stream_ptr(stream)))


GEMM_SYMMETRIC = 1
GEMM_PAIR = 2


def gemm(a, b, out, aux=None, b_mn_major: bool = False, alpha: float = 1.0, beta: float = 0.0,
         diag: float = 0.0, symmetric: bool = False, pair: bool = False, scratch=None,
         stream=None) -> None:
    """out = alpha * a @ op(b) + beta * aux + diag * I on the tensor-core engine.

    ``a`` is M x K; ``b`` is N x K (op = transpose) or, with ``b_mn_major``, K x N.  All
    tensors are 2D bf16 or all fp16, with unit column stride.  ``symmetric`` declares the
    result symmetric: the upper triangle is computed and mirrored.  ``pair`` runs the 2-SM
    kernel (256 x 256 tiles on clusters of two CTAs)."""
    import torch
    M, K = a.shape
    N = b.shape[1] if b_mn_major else b.shape[0]
    fp16 = 1 if a.dtype == torch.float16 else 0
    flags = (GEMM_SYMMETRIC if symmetric else 0) | (GEMM_PAIR if pair else 0)
    if scratch is None:
        need = lib().nsm_gemm_scratch_bytes(M, N, flags)
        scratch = torch.empty(max(int(need), 1024), dtype=torch.uint8, device=a.device)
    _check(lib().nsm_gemm(_ptr(a), a.stride(0), _ptr(b), b.stride(0), _ptr(out), out.stride(0),
                          _ptr(aux), 0 if aux is None else aux.stride(0), M, N, K,
                          1 if b_mn_major else 0, fp16, flags, float(alpha), float(beta),
                          float(diag), _ptr(scratch), scratch.numel(), _stream_ptr(stream)))


def device_status(stream=None) -> int:
    """Synchronises the stream; returns NSM_OK, NSM_ERR_TIMEOUT or (checked build)
    NSM_ERR_BOUNDS, and clears the record."""
    v = ctypes.c_int(0)
    _check(lib().nsm_device_status(_stream_ptr(stream), ctypes.byref(v)))
    return v.value


def device_status_detail(stream=None) -> Tuple[int, int, int, int]:
    """Synchronises the stream; returns (status, kernel, role, site) of the first bounded
    wait that expired, or (checked build) bounds test that failed, since the last read
    (status NSM_OK and zeros when none), and clears the record.  kernel/role/site are the
    NSM_KERNEL_* / NSM_ROLE_* / NSM_SITE_* codes of the C header."""
    v = [ctypes.c_int(0) for _ in range(4)]
    _check(lib().nsm_device_status_detail(_stream_ptr(stream), *[ctypes.byref(x) for x in v]))
    return tuple(x.value for x in v)


NSM_KERNEL_GEMM, NSM_KERNEL_GEMM_PAIR, NSM_KERNEL_SMALL, NSM_KERNEL_SELFTEST = 1, 2, 3, 4
NSM_SITE_SELFTEST = 11
NSM_SITE_SELFTEST_BOUNDS = 23

OPT_PAIR_KERNELS, OPT_SMALL_KERNEL, OPT_PDL, OPT_BOUNDS_CHECKS, OPT_SYM_STORAGE = 1, 2, 3, 4, 5


def set_option(option: int, value: int) -> None:
    """Process-wide choice between the library's equivalent paths (for comparisons):
    OPT_PAIR_KERNELS, OPT_SMALL_KERNEL, OPT_SYM_STORAGE (default 1: symmetric iterates
    kept as their upper 256 x 256 tiles where every launch is on the 2-SM kernel) and
    OPT_PDL (0 off, 1 on, default 2: on for tables of at most 2^25 elements)."""
    _check(lib().nsm_set_option(int(option), int(value)))


def get_option(option: int) -> int:
    return _check(lib().nsm_get_option(int(option)))


def status_selftest(wait_us: int = 20000, stream=None) -> None:
    """Launches one CTA whose bounded wait expires after wait_us and records a timeout in
    the device status word (read it with device_status)."""
    _check(lib().nsm_status_selftest(int(wait_us), _stream_ptr(stream)))


def bounds_selftest(stream=None) -> None:
    """Launches one thread that runs the kernels' bounds test on an index past its range
    and makes no access: the checked build records NSM_ERR_BOUNDS (read it with
    device_status_detail), the regular build nothing."""
    _check(lib().nsm_bounds_selftest(_stream_ptr(stream)))


def copy_to_device(dst, src, stream=None, ctas: int = 0) -> None:
    """dst (device tensor) <- src (pinned host tensor of the same byte size) by SM loads
    over the host link (nsm_copy_to_device); asynchronous on `stream`."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src differ in size")
    _check(lib().nsm_copy_to_device(_ptr(dst), _ptr(src), nbytes, int(ctas), _stream_ptr(stream)))


def checked_build() -> bool:
    """Whether the loaded library is the bounds-checked build."""
    return get_option(OPT_BOUNDS_CHECKS) == 1


def timing_enable(on: bool = True) -> None:
    lib().nsm_timing_enable(1 if on else 0)


def timing_reset() -> None:
    lib().nsm_timing_reset()


KIND_GEMM, KIND_MOMENTUM, KIND_NORM, KIND_LAYOUT, KIND_APPLY, KIND_ADAMW, KIND_SMALL, KIND_GRAD_NORM = range(8)
KIND_NAMES = {KIND_GEMM: "k_ns_gemm", KIND_MOMENTUM: "k_momentum_class", KIND_NORM: "k_scale_finalize",
              KIND_LAYOUT: "k_to_class", KIND_APPLY: "k_from_class", KIND_ADAMW: "k_adamw",
              KIND_SMALL: "k_ns_small", KIND_GRAD_NORM: "k_grad_norm"}


def timing_read(kind: int = KIND_GEMM) -> Tuple[float, int, float]:
    """(device ms, launches, algorithmic work) of one kernel kind since the last reset."""
    ms = ctypes.c_double(0)
    n = ctypes.c_int64(0)
    w = ctypes.c_double(0)
    _check(lib().nsm_timing_read_kind(int(kind), ctypes.byref(ms), ctypes.byref(n), ctypes.byref(w)))
    return ms.value, n.value, w.value


# ---------------------------------------------------------------- optimizer wrapper

class MuonAdamW:
    """Hybrid optimizer state over named parameters, on one GPU.

    Parameters tagged by :func:`route` go to one packed Muon group (fp32 master params,
    fp32 momentum, a bf16 gradient buffer); the rest go to one flat AdamW group (fp32
    master params and moments, bf16 gradients).  The config keys mirror the pages:
    ``muon_lr`` / ``adam_lr`` override ``lr``, ``momentum``, ``weight_decay``, ``betas``,
    ``eps`` and ``ns_method``.  The optimizer owns the fp32 master weights: callers write
    initial weights and each step's gradients through :meth:`param` / :meth:`grad`, and
    :meth:`state_dict` carries the master weights with the moments, so that a checkpoint
    restores the whole state.
    """

    def __init__(self, named_shapes: Iterable[Tuple[str, Tuple[int, ...]]], device="cuda",
                 lr: Optional[float] = None, muon_lr: Optional[float] = None,
                 adam_lr: Optional[float] = None, momentum: float = MUON_MOMENTUM_DEFAULT,
                 weight_decay: float = 0.0, betas=ADAM_BETAS_DEFAULT,
                 eps: float = ADAM_EPS_DEFAULT, ns_method: str = NS_METHOD_DEFAULT,
                 ns_steps: int = NS_STEPS_DEFAULT, nesterov: bool = True):
        import torch
        named = list(named_shapes)
        self.muon_names: List[str] = []
        self.muon_shapes: List[Tuple[int, int]] = []
        self.adam_names: List[str] = []
        self.adam_sizes: List[int] = []
        self._shape_of: Dict[str, Tuple[int, ...]] = {}
        for name, shape in named:
            shape = tuple(int(d) for d in shape)
            if name in self._shape_of:
                raise ValueError(f"parameter {name!r} is listed twice")
            self._shape_of[name] = shape
            if route(name, len(shape)):
                cols = 1
                for d in shape[1:]:
                    cols *= d
                self.muon_names.append(name)
                self.muon_shapes.append((shape[0], cols))
            else:
                size = 1
                for d in shape:
                    size *= d
                self.adam_names.append(name)
                self.adam_sizes.append(size)
        base_lr = lr
        self.muon_lr = muon_lr if muon_lr is not None else (base_lr if base_lr is not None else MUON_LR_DEFAULT)
        self.adam_lr = adam_lr if adam_lr is not None else (base_lr if base_lr is not None else ADAM_LR_DEFAULT)
        self.momentum = momentum
        self.weight_decay = weight_decay
        self.betas = tuple(betas)
        self.eps = eps
        self.ns_method = ns_method
        self.ns_steps = ns_steps
        self.nesterov = nesterov
        self.step_count = 0
        dev = torch.device(device)
        self._muon_index = {n: i for i, n in enumerate(self.muon_names)}
        self._adam_offset: Dict[str, int] = {}
        off = 0
        for n, size in zip(self.adam_names, self.adam_sizes):
            self._adam_offset[n] = off
            off += size
        if self.muon_shapes:
            self.offsets, total = pack(self.muon_shapes)
            self.muon_params = torch.zeros(total, dtype=torch.float32, device=dev)
            self.muon_momentum = torch.zeros(total, dtype=torch.float32, device=dev)
            self.muon_grads = torch.zeros(total, dtype=torch.bfloat16, device=dev)
            self.workspace = torch.empty(workspace_bytes(self.muon_shapes, ns_method, ns_steps),
                                         dtype=torch.uint8, device=dev)
        n_adam = sum(self.adam_sizes)
        self.adam_params = torch.zeros(n_adam, dtype=torch.float32, device=dev)
        self.adam_exp_avg = torch.zeros(n_adam, dtype=torch.float32, device=dev)
        self.adam_exp_avg_sq = torch.zeros(n_adam, dtype=torch.float32, device=dev)
        self.adam_grads = torch.zeros(n_adam, dtype=torch.bfloat16, device=dev)

    def _view(self, name: str, muon_buf, adam_buf):
        shape = self._shape_of[name]
        if name in self._muon_index:
            i = self._muon_index[name]
            r, c = self.muon_shapes[i]
            o = int(self.offsets[i])
            return muon_buf[o:o + r * c].view(shape)
        o = self._adam_offset[name]
        size = 1
        for d in shape:
            size *= d
        return adam_buf[o:o + size].view(shape)

    def param(self, name: str):
        """The fp32 master weight of a parameter (a view into its group's buffer)."""
        return self._view(name, getattr(self, "muon_params", None), self.adam_params)

    def grad(self, name: str):
        """The bf16 gradient slot of a parameter (a view; write each step's gradient here)."""
        return self._view(name, getattr(self, "muon_grads", None), self.adam_grads)

    def step(self, stream=None) -> None:
        self.step_count += 1
        if self.muon_shapes:
            muon_step(self.muon_grads, self.muon_params, self.muon_momentum, self.offsets,
                      self.muon_shapes, self.muon_lr, self.weight_decay, self.momentum,
                      self.ns_method, self.ns_steps, self.nesterov, self.workspace, stream)
        if self.adam_params.numel():
            adamw_step(self.adam_grads, self.adam_params, self.adam_exp_avg, self.adam_exp_avg_sq,
                       self.adam_lr, self.betas[0], self.betas[1], self.eps, self.weight_decay,
                       self.step_count, stream)

    def state_dict(self) -> Dict[str, object]:
        """The whole optimizer state as plain tensors (the caller saves and restores them):
        the step count, both groups' fp32 master weights, the Muon momentum and the AdamW
        moments, with the names and shapes they were packed from."""
        d: Dict[str, object] = {"step": self.step_count,
                                "muon_names": list(self.muon_names),
                                "muon_shapes": list(self.muon_shapes),
                                "adam_names": list(self.adam_names),
                                "adam_sizes": list(self.adam_sizes),
                                "adam_params": self.adam_params,
                                "adam_exp_avg": self.adam_exp_avg,
                                "adam_exp_avg_sq": self.adam_exp_avg_sq}
        if self.muon_shapes:
            d["muon_params"] = self.muon_params
            d["muon_momentum"] = self.muon_momentum
        return d

    def load_state_dict(self, d: Dict[str, object]) -> None:
        if (list(d["muon_names"]) != self.muon_names or list(d["adam_names"]) != self.adam_names
                or [tuple(s) for s in d["muon_shapes"]] != self.muon_shapes
                or list(d["adam_sizes"]) != self.adam_sizes):
            raise ValueError("state_dict was saved for other parameters")
        self.step_count = int(d["step"])
        self.adam_params.copy_(d["adam_params"])
        self.adam_exp_avg.copy_(d["adam_exp_avg"])
        self.adam_exp_avg_sq.copy_(d["adam_exp_avg_sq"])
        if self.muon_shapes:
            self.muon_params.copy_(d["muon_params"])
            self.muon_momentum.copy_(d["muon_momentum"])
