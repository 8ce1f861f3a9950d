"""Python binding of the C ABI in ``include/mla_decode.h`` (ctypes).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  PyTorch tensors supply device memory and the current stream;
their data pointers are handed to the library unchanged.  There is no
fallback path: if the compiled library is missing, loading it raises.

The plan / run split, and the plan arguments (head_dim_ckv = kv_lora_rank,
head_dim_kpe = qk_rope_head_dim, page_size, sm_scale, no causal mask), follow
the decode_wrapper.plan call reviewed in "[WIP] support flashinfer_mla"
(vLLM-metax PR #113).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libmla_decode.so")

# mla_status_t
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CAPACITY, ERR_CUDA, ERR_DEVICE_TIMEOUT, \
    ERR_DEVICE_BOUNDS, ERR_NOT_PLANNED = range(8)
# mla_dtype_t
DTYPE_BF16, DTYPE_FP8_E4M3, DTYPE_FP32 = 0, 1, 2
# mla_kernel_t
KERNEL_DEFAULT, KERNEL_TCGEN05, KERNEL_MMA_SYNC, KERNEL_PAIR = 0, 1, 2, 3
KERNELS = {"default": KERNEL_DEFAULT, "tcgen05": KERNEL_TCGEN05, "mma_sync": KERNEL_MMA_SYNC,
           "pair": KERNEL_PAIR}

EXPORTED = ("mla_plan_create", "mla_decode_plan", "mla_decode_run", "mla_decode_run_host",
            "mla_plan_check_status", "mla_plan_info", "mla_plan_destroy", "mla_status_string",
            "mla_plan_last_error", "mla_plan_partition_host", "mla_plan_set_profile_events",
            "mla_decode_noalloc", "mla_decode_plan_multi", "mla_merge_states",
            "mla_absorb_q", "mla_project_out")


class MLAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("num_workers", ctypes.c_int32),
                ("num_units", ctypes.c_int32), ("num_partial_slots", ctypes.c_int32),
                ("num_merge", ctypes.c_int32), ("total_tiles", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("tile_tokens", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None
_I32P = ctypes.POINTER(ctypes.c_int32)
_VP = ctypes.c_void_p


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = bind_library(path)
    return _lib


def bind_library(path: str) -> ctypes.CDLL:
    """Open a build of the library at ``path`` and declare the C signatures
    on it (a separate handle; the module's own calls keep using
    ``load_library``'s)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "paged_mla_decode_02_gb300.build.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    c_int, c_float = ctypes.c_int, ctypes.c_float
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [c_int]
    lib.mla_plan_last_error.restype = ctypes.c_char_p
    lib.mla_plan_last_error.argtypes = [_VP]
    lib.mla_plan_create.restype = c_int
    lib.mla_plan_create.argtypes = [c_int, c_int, c_int, ctypes.POINTER(_VP)]
    lib.mla_plan_destroy.restype = c_int
    lib.mla_plan_destroy.argtypes = [_VP]
    lib.mla_decode_plan.restype = c_int
    lib.mla_decode_plan.argtypes = [_VP, _I32P, _VP, _I32P, c_int, c_int, c_int, c_int, c_int,
                                    c_float, _VP]
    lib.mla_absorb_q.restype = c_int
    lib.mla_absorb_q.argtypes = [_VP, _VP, _VP, c_int, c_int, c_int, c_int, _VP]
    lib.mla_project_out.restype = c_int
    lib.mla_project_out.argtypes = [_VP, _VP, _VP, c_int, c_int, c_int, c_int, _VP]
    lib.mla_merge_states.restype = c_int
    lib.mla_merge_states.argtypes = [_VP, _VP, _VP, _VP, _VP, c_int, _VP, c_int, _VP]
    lib.mla_decode_plan_multi.restype = c_int
    lib.mla_decode_plan_multi.argtypes = [_VP, _I32P, _VP, _I32P, c_int, c_int, c_int, c_int,
                                          c_int, c_int, c_float, _VP]
    lib.mla_decode_run.restype = c_int
    lib.mla_decode_run.argtypes = [_VP, _VP, _VP, c_int, _VP, _VP, c_int, c_float, c_int, _VP,
                                   c_int, _VP, _VP]
    lib.mla_decode_run_host.restype = c_int
    lib.mla_decode_run_host.argtypes = lib.mla_decode_run.argtypes
    lib.mla_plan_check_status.restype = c_int
    lib.mla_plan_check_status.argtypes = [_VP]
    lib.mla_plan_info.restype = c_int
    lib.mla_plan_info.argtypes = [_VP, ctypes.POINTER(PlanInfo)]
    lib.mla_plan_set_profile_events.restype = c_int
    lib.mla_plan_set_profile_events.argtypes = [_VP, _VP, _VP]
    lib.mla_plan_partition_host.restype = c_int
    lib.mla_plan_partition_host.argtypes = [_I32P, _I32P, c_int, c_int, c_int, c_int, c_float,
                                            c_int, c_int, _I32P, c_int, _I32P, _I32P, c_int,
                                            _I32P]
    lib.mla_decode_noalloc.restype = c_int
    lib.mla_decode_noalloc.argtypes = [_I32P, _VP, _I32P, c_int, c_int, c_int, c_float, _VP, _VP,
                                       _VP, _VP, c_float, c_int, _VP, c_int, _VP, c_int, _VP]
    return lib


def status_string(status: int) -> str:
    return load_library().mla_status_string(status).decode()


def _check(status: int, plan=None, what: str = "") -> None:
    if status != OK:
        lib = load_library()
        detail = lib.mla_plan_last_error(plan).decode() if plan else ""
        msg = f"{what}: {status_string(status)}"
        if detail:
            msg += f" ({detail})"
        raise MLAError(status, msg)


def _i32_host(a) -> np.ndarray:
    """A contiguous host int32 array from a numpy array, list or CPU tensor."""
    if hasattr(a, "detach"):
        if a.device.type != "cpu":
            raise ValueError("kv_indptr / kv_len must be host (CPU) arrays")
        a = a.detach().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(t) -> int:
    return int(t.data_ptr())


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t, what: str) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return DTYPE_FP8_E4M3
    raise ValueError(f"{what}: unsupported dtype {t.dtype}")


# ---------------------------------------------------------------------------
# The C ABI entry points, under the same names
# ---------------------------------------------------------------------------

def mla_plan_create(max_batch: int, num_heads: int, kernel="default") -> int:
    """Create a plan on the current CUDA device; returns an opaque handle."""
    lib = load_library()
    handle = _VP()
    k = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    _check(lib.mla_plan_create(int(max_batch), int(num_heads), k, ctypes.byref(handle)), None,
           "mla_plan_create")
    return handle.value


def mla_plan_destroy(plan) -> None:
    if plan:
        load_library().mla_plan_destroy(plan)


def mla_decode_plan(plan, kv_indptr, kv_indices, kv_len, num_heads: int, head_dim_ckv: int,
                    head_dim_kpe: int, page_size: int, sm_scale: float, stream=None) -> None:
    """Plan one batch.  kv_indptr / kv_len are HOST int32 arrays, kv_indices a
    device int32 tensor that must stay alive until the plan's last run."""
    lib = load_library()
    indptr = _i32_host(kv_indptr)
    lens = _i32_host(kv_len)
    batch = lens.shape[0]
    if indptr.shape[0] != batch + 1:
        raise ValueError("kv_indptr must have batch + 1 entries")
    idx_ptr = _ptr(kv_indices) if kv_indices is not None and kv_indices.numel() > 0 else None
    st = lib.mla_decode_plan(plan, indptr.ctypes.data_as(_I32P), idx_ptr,
                             lens.ctypes.data_as(_I32P), batch, int(num_heads),
                             int(head_dim_ckv), int(head_dim_kpe), int(page_size),
                             float(sm_scale), _stream_handle(stream))
    _check(st, plan, "mla_decode_plan")


def mla_decode_plan_multi(plan, kv_indptr, kv_indices, kv_len, q_len: int, num_heads: int,
                          head_dim_ckv: int, head_dim_kpe: int, page_size: int, sm_scale: float,
                          stream=None) -> None:
    """Plan a step of q_len query tokens per request (causal inside the query
    block; see mla_decode.h).  Arrays as for ``mla_decode_plan``."""
    lib = load_library()
    indptr = _i32_host(kv_indptr)
    lens = _i32_host(kv_len)
    batch = lens.shape[0]
    if indptr.shape[0] != batch + 1:
        raise ValueError("kv_indptr must have batch + 1 entries")
    idx_ptr = _ptr(kv_indices) if kv_indices is not None and kv_indices.numel() > 0 else None
    st = lib.mla_decode_plan_multi(plan, indptr.ctypes.data_as(_I32P), idx_ptr,
                                   lens.ctypes.data_as(_I32P), batch, int(q_len), int(num_heads),
                                   int(head_dim_ckv), int(head_dim_kpe), int(page_size),
                                   float(sm_scale), _stream_handle(stream))
    _check(st, plan, "mla_decode_plan_multi")


def _bf16_contig(name, t):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 tensor")


def mla_absorb_q(q_raw, w_uk, q_nope=None, check_status: bool = False, stream=None):
    """q_nope[b,h] = W_UK[h] . q_raw[b,h]: q_raw bf16 [B,H,dn], w_uk bf16
    [H,512,dn]; returns (or fills) q_nope bf16 [B,H,512]."""
    import torch
    B, H, dn = q_raw.shape
    if q_nope is None:
        q_nope = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q_raw.device)
    for name, t in (("q_raw", q_raw), ("w_uk", w_uk), ("q_nope", q_nope)):
        _bf16_contig(name, t)
    if tuple(w_uk.shape) != (H, 512, dn) or tuple(q_nope.shape) != (B, H, 512):
        raise ValueError("w_uk must be [H, 512, dn] and q_nope [B, H, 512]")
    st = load_library().mla_absorb_q(_ptr(q_raw), _ptr(w_uk), _ptr(q_nope), B, H, dn,
                                     int(bool(check_status)), _stream_handle(stream))
    _check(st, None, "mla_absorb_q")
    return q_nope


def mla_project_out(out, w_uv, o=None, check_status: bool = False, stream=None):
    """o[b,h] = out[b,h] . W_UV[h]: out bf16 [B,H,512], w_uv bf16 [H,512,dv];
    returns (or fills) o bf16 [B,H,dv]."""
    import torch
    B, H, _ = out.shape
    dv = w_uv.shape[2]
    if o is None:
        o = torch.empty((B, H, dv), dtype=torch.bfloat16, device=out.device)
    for name, t in (("out", out), ("w_uv", w_uv), ("o", o)):
        _bf16_contig(name, t)
    if tuple(out.shape) != (B, H, 512) or tuple(w_uv.shape) != (H, 512, dv) or tuple(o.shape) != (B, H, dv):
        raise ValueError("out must be [B, H, 512], w_uv [H, 512, dv] and o [B, H, dv]")
    st = load_library().mla_project_out(_ptr(out), _ptr(w_uv), _ptr(o), B, H, dv,
                                        int(bool(check_status)), _stream_handle(stream))
    _check(st, None, "mla_project_out")
    return o


def mla_merge_states(o_a, lse_a, o_b, lse_b, out, lse_out, stream=None) -> None:
    """Combine two attention states of the same rows over disjoint token sets
    by log-sum-exp (see mla_decode.h).  o_a / o_b fp32 [..., 512], lse_a /
    lse_b fp32 [...] on the device; out (bf16 or fp32) and lse_out may alias
    the inputs."""
    import torch
    lib = load_library()
    rows = int(lse_a.numel())
    for name, t in (("o_a", o_a), ("o_b", o_b), ("out", out)):
        if not t.is_contiguous() or t.numel() != rows * 512:
            raise ValueError(f"{name} must be a contiguous [rows, 512] tensor")
    for name, t in (("o_a", o_a), ("o_b", o_b), ("lse_a", lse_a), ("lse_b", lse_b), ("lse_out", lse_out)):
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    if lse_b.numel() != rows or lse_out.numel() != rows:
        raise ValueError("lse tensors must have one entry per row")
    st = lib.mla_merge_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(out),
                              _dtype_code(out, "out"), _ptr(lse_out), rows, _stream_handle(stream))
    _check(st, None, "mla_merge_states")


def _check_layouts(q_nope, q_pe, ckv_cache, kpe_cache, out, lse, page_size=None) -> None:
    """The shapes mla_decode.h documents, checked before the library reads
    through the raw pointers: the cache [pages, page_size, 512] and [pages,
    page_size, 64] of one dtype, q [..., 512] / [..., 64], out [..., 512] and
    lse [...] over the same leading dims."""
    if ckv_cache.dim() != 3 or ckv_cache.shape[2] != 512:
        raise ValueError(f"ckv_cache must be [num_pages, page_size, 512], got {tuple(ckv_cache.shape)}")
    if tuple(kpe_cache.shape) != (ckv_cache.shape[0], ckv_cache.shape[1], 64):
        raise ValueError(f"kpe_cache must be [num_pages, page_size, 64] like ckv_cache, "
                         f"got {tuple(kpe_cache.shape)}")
    if kpe_cache.dtype != ckv_cache.dtype:
        raise ValueError("ckv_cache and kpe_cache must have the same dtype")
    if page_size is not None and ckv_cache.shape[1] != page_size:
        raise ValueError(f"the cache holds pages of {ckv_cache.shape[1]} tokens, the plan {page_size}")
    lead = tuple(q_nope.shape[:-1])
    if q_nope.shape[-1] != 512 or tuple(q_pe.shape) != lead + (64,):
        raise ValueError("q_nope must be [..., 512] and q_pe [..., 64] over the same leading dims")
    if tuple(out.shape) != lead + (512,) or tuple(lse.shape) != lead:
        raise ValueError("out must be [..., 512] and lse [...] over q_nope's leading dims")


def mla_decode_run(plan, q_nope, q_pe, ckv_cache, kpe_cache, out, lse, kv_scale: float = 1.0,
                   stream=None, page_size=None) -> None:
    """Run the planned batch on device tensors (see mla_decode.h for layouts)."""
    lib = load_library()
    for name, t in (("q_nope", q_nope), ("q_pe", q_pe), ("ckv_cache", ckv_cache),
                    ("kpe_cache", kpe_cache), ("out", out), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    _check_layouts(q_nope, q_pe, ckv_cache, kpe_cache, out, lse, page_size)
    num_pages = int(ckv_cache.shape[0])
    st = lib.mla_decode_run(plan, _ptr(q_nope), _ptr(q_pe), _dtype_code(q_nope, "q_nope"),
                            _ptr(ckv_cache), _ptr(kpe_cache), _dtype_code(ckv_cache, "ckv_cache"),
                            float(kv_scale), num_pages, _ptr(out), _dtype_code(out, "out"),
                            _ptr(lse), _stream_handle(stream))
    _check(st, plan, "mla_decode_run")


def mla_decode_noalloc(kv_indptr, kv_indices, kv_len, page_size: int, sm_scale: float, q_nope,
                       q_pe, ckv_cache, kpe_cache, out, lse, kv_scale: float = 1.0,
                       check_status: bool = True, stream=None) -> None:
    """Plan + run one batch from the library's fixed scratch memory: the call
    allocates no device memory (out / lse are the caller's tensors).  Calls
    must not overlap; see mla_decode.h for the limits."""
    lib = load_library()
    indptr = _i32_host(kv_indptr)
    lens = _i32_host(kv_len)
    batch = lens.shape[0]
    if indptr.shape[0] != batch + 1:
        raise ValueError("kv_indptr must have batch + 1 entries")
    for name, t in (("q_nope", q_nope), ("q_pe", q_pe), ("ckv_cache", ckv_cache),
                    ("kpe_cache", kpe_cache), ("out", out), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if _dtype_code(q_nope, "q_nope") != DTYPE_BF16 or _dtype_code(ckv_cache, "ckv_cache") != DTYPE_BF16:
        raise ValueError("mla_decode_noalloc takes bf16 queries and caches")
    _check_layouts(q_nope, q_pe, ckv_cache, kpe_cache, out, lse, int(page_size))
    idx_ptr = _ptr(kv_indices) if kv_indices is not None and kv_indices.numel() > 0 else None
    st = lib.mla_decode_noalloc(indptr.ctypes.data_as(_I32P), idx_ptr, lens.ctypes.data_as(_I32P),
                                batch, int(q_nope.shape[1]), int(page_size), float(sm_scale),
                                _ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
                                float(kv_scale), int(ckv_cache.shape[0]), _ptr(out),
                                _dtype_code(out, "out"), _ptr(lse), int(bool(check_status)),
                                _stream_handle(stream))
    _check(st, None, "mla_decode_noalloc")


def mla_decode_run_host(plan, q_nope_host, q_pe_host, ckv_cache, kpe_cache, out_host, lse_host,
                        kv_scale: float = 1.0, stream=None) -> None:
    """One decode step from host q buffers to host out / lse (the cache stays on the device)."""
    lib = load_library()
    for name, t in (("q_nope", q_nope_host), ("q_pe", q_pe_host), ("out", out_host),
                    ("lse", lse_host)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    if not ckv_cache.is_cuda or not kpe_cache.is_cuda:
        raise ValueError("the cache must be on the device")
    _check_layouts(q_nope_host, q_pe_host, ckv_cache, kpe_cache, out_host, lse_host)
    st = lib.mla_decode_run_host(plan, _ptr(q_nope_host), _ptr(q_pe_host),
                                 _dtype_code(q_nope_host, "q_nope"), _ptr(ckv_cache),
                                 _ptr(kpe_cache), _dtype_code(ckv_cache, "ckv_cache"),
                                 float(kv_scale), int(ckv_cache.shape[0]), _ptr(out_host),
                                 _dtype_code(out_host, "out"), _ptr(lse_host),
                                 _stream_handle(stream))
    _check(st, plan, "mla_decode_run_host")


def mla_plan_check_status(plan) -> int:
    """Synchronise and return the device status (raises on a device error)."""
    st = load_library().mla_plan_check_status(plan)
    _check(st, plan, "mla_plan_check_status")
    return st


def mla_plan_set_profile_events(plan, start_event, stop_event) -> None:
    """Record torch.cuda.Event start/stop around the decode kernel of every run (None: off)."""
    h0 = int(start_event.cuda_event) if start_event is not None else None
    h1 = int(stop_event.cuda_event) if stop_event is not None else None
    _check(load_library().mla_plan_set_profile_events(plan, h0, h1), plan,
           "mla_plan_set_profile_events")


def mla_plan_info(plan) -> dict:
    info = PlanInfo()
    _check(load_library().mla_plan_info(plan, ctypes.byref(info)), plan, "mla_plan_info")
    return info.as_dict()


def mla_plan_partition_host(kv_indptr, kv_len, num_workers: int, tile_tokens: int,
                            page_size: int, head_dim_ckv: int = 512, head_dim_kpe: int = 64,
                            sm_scale: float = 1.0):
    """The host planner alone: returns (units [n,6], worker_ptr [W+1], merge [m,3], n_slots)."""
    lib = load_library()
    indptr = _i32_host(kv_indptr)
    lens = _i32_host(kv_len)
    batch = lens.shape[0]
    ucap = num_workers + batch
    units = np.zeros((ucap, 6), np.int32)
    wptr = np.zeros(num_workers + 1, np.int32)
    merge = np.zeros((batch, 3), np.int32)
    counts = np.zeros(3, np.int32)
    st = lib.mla_plan_partition_host(indptr.ctypes.data_as(_I32P), lens.ctypes.data_as(_I32P),
                                     batch, head_dim_ckv, head_dim_kpe, page_size, sm_scale,
                                     num_workers, tile_tokens, units.ctypes.data_as(_I32P), ucap,
                                     wptr.ctypes.data_as(_I32P), merge.ctypes.data_as(_I32P),
                                     batch, counts.ctypes.data_as(_I32P))
    if st != OK:
        raise MLAError(st, f"mla_plan_partition_host: {status_string(st)}")
    return units[:counts[0]].copy(), wptr, merge[:counts[2]].copy(), int(counts[1])


# ---------------------------------------------------------------------------
# Convenience wrapper
# ---------------------------------------------------------------------------

class MLADecoder:
    """Owns one plan: ``plan(...)`` once per batch layout, ``run(...)`` per step."""

    def __init__(self, max_batch: int, num_heads: int, kernel="default"):
        self.num_heads = int(num_heads)
        self.handle = mla_plan_create(max_batch, num_heads, kernel)
        self._kv_indices = None
        self.page_size = None

    def plan(self, kv_indptr, kv_indices, kv_len, page_size: int, sm_scale: float,
             head_dim_ckv: int = 512, head_dim_kpe: int = 64, stream=None, q_len: int = 0) -> None:
        """q_len 0: one query token per request (q and out [B, H, .]);
        q_len >= 1: that many, causal inside the block (q and out [B, Q, H, .])."""
        if q_len:
            mla_decode_plan_multi(self.handle, kv_indptr, kv_indices, kv_len, q_len,
                                  self.num_heads, head_dim_ckv, head_dim_kpe, page_size,
                                  sm_scale, stream)
        else:
            mla_decode_plan(self.handle, kv_indptr, kv_indices, kv_len, self.num_heads,
                            head_dim_ckv, head_dim_kpe, page_size, sm_scale, stream)
        self.q_len = int(q_len)
        self.page_size = int(page_size)
        self._kv_indices = kv_indices     # keep the borrowed page table alive

    def run(self, q_nope, q_pe, ckv_cache, kpe_cache, out=None, lse=None,
            kv_scale: float = 1.0, out_dtype=None, stream=None):
        import torch
        lead = tuple(q_nope.shape[:-1])          # (B, H) or (B, Q, H)
        if out is None:
            out = torch.empty(lead + (512,), dtype=out_dtype or torch.bfloat16, device=q_nope.device)
        if lse is None:
            lse = torch.empty(lead, dtype=torch.float32, device=q_nope.device)
        mla_decode_run(self.handle, q_nope, q_pe, ckv_cache, kpe_cache, out, lse, kv_scale, stream,
                       page_size=self.page_size)
        return out, lse

    def info(self) -> dict:
        return mla_plan_info(self.handle)

    def check_status(self) -> int:
        return mla_plan_check_status(self.handle)

    def close(self) -> None:
        if self.handle:
            mla_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
