"""Python binding of libsmla_l1norm (GB300 Sparse-Flash-MLA Softmax-L1Norm forward).

Argument marshalling only: every step of the operator runs in the CUDA
library.  The names follow the C ABI in ``include/smla_l1norm.h``; tensors
are passed as torch CUDA tensors (their device pointers go to the library)
and streams as torch streams.  There is no CPU path: without the built
library every call raises.

Operator (article "SparseFlashMlaSoftmaxL1Norm", CANN ops-transformer,
section 三阶段计算公式)::

    out[row, i] = (1/G) * sum_g exp(scale * q[row, g] . K[j_i] - lse[row, g])

over the slots kept by the mask (0 elsewhere), j_i = sparse_indices[row, i]
or i in the dense form.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import build as _build

__all__ = [
    "SMLA_OK", "SMLA_ERR_NULLPTR", "SMLA_ERR_INVALID", "SMLA_ERR_UNSUPPORTED", "SMLA_ERR_CUDA",
    "SMLA_ERR_TIMEOUT", "SMLA_WARN_BAD_INDEX", "SMLA_ERR_CAPACITY", "SmlaError", "Plan", "library",
    "library_path", "sparse_flash_mla_softmax_l1_norm", "schedule_host", "wait_timeout_probe",
    "run_noalloc", "noalloc_config",
]

SMLA_OK, SMLA_ERR_NULLPTR, SMLA_ERR_INVALID, SMLA_ERR_UNSUPPORTED = 0, 1, 2, 3
SMLA_ERR_CUDA, SMLA_ERR_TIMEOUT, SMLA_WARN_BAD_INDEX, SMLA_ERR_CAPACITY = 4, 5, 6, 7
LAYOUTS = {"BSND": 0, "TND": 1}
DTYPES = {"fp16": 0, "float16": 0, "bf16": 1, "bfloat16": 1}


class SmlaError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str = ""):
        self.code = code
        msg = f"{what}: {library().smla_status_string(code).decode()}"
        if detail:
            msg += f" [{detail}]"
        super().__init__(msg)


class _Desc(ctypes.Structure):
    _fields_ = [
        ("layout_q", ctypes.c_int32), ("layout_k", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32), ("num_heads_k", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("batch_size", ctypes.c_int32), ("max_seqlen_q", ctypes.c_int32), ("max_seqlen_k", ctypes.c_int32),
        ("topk", ctypes.c_int32), ("mask_mode", ctypes.c_int32), ("cmp_ratio", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float), ("has_topk_length", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int32)), ("cu_seqlens_k", ctypes.POINTER(ctypes.c_int32)),
        ("topk_length_hint", ctypes.POINTER(ctypes.c_int32)), ("num_ctas", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int64), ("num_items", ctypes.c_int64), ("num_ctas", ctypes.c_int32),
        ("rows_per_item", ctypes.c_int32), ("mma_n", ctypes.c_int32), ("stages", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32), ("out_width", ctypes.c_int32), ("est_tiles", ctypes.c_int64),
        ("max_cta_cost", ctypes.c_double), ("mean_cta_cost", ctypes.c_double),
        ("q_rows_total", ctypes.c_int64), ("k_rows_total", ctypes.c_int64),
        ("host_chunks", ctypes.c_int32), ("mma_issuers", ctypes.c_int32), ("cta_pairs", ctypes.c_int32),
        ("split_tiles", ctypes.c_int32), ("split_items", ctypes.c_int64),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class _Tensors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("q", "k", "softmax_lse", "sparse_indices", "topk_length", "seqused_q", "seqused_k", "out",
                 "cmp_residual_k")]


class IoSizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("q_bytes", "k_bytes", "lse_bytes", "indices_bytes", "topk_length_bytes", "out_bytes")]


_LIB = None


def library_path() -> str:
    return _build.LIB


def library():
    """Load the built library (building it first if the sources are newer)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if not os.path.exists(path) or _build.sources_newer_than(path):
        try:
            path = _build.build()
        except Exception as e:  # no silent fallback: the operator only exists in CUDA
            raise RuntimeError(f"softmax_l1_norm_gb300: CUDA library unavailable ({e})") from e
    lib = ctypes.CDLL(path)
    P, I32, I64, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.smla_l1norm_plan_create.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(P)]
    lib.smla_l1norm_plan_create.restype = I32
    lib.smla_l1norm_plan_destroy.argtypes = [P]
    lib.smla_l1norm_plan_destroy.restype = None
    lib.smla_l1norm_output_shape.argtypes = [P, ctypes.POINTER(I64), ctypes.POINTER(I32)]
    lib.smla_l1norm_output_shape.restype = I32
    lib.smla_l1norm_plan_get_info.argtypes = [P, ctypes.POINTER(PlanInfo)]
    lib.smla_l1norm_plan_get_info.restype = I32
    lib.smla_l1norm_run.argtypes = [P, P, P, P, P, P, P, P]
    lib.smla_l1norm_run.restype = I32
    lib.smla_l1norm_run_tensors.argtypes = [P, ctypes.POINTER(_Tensors), P]
    lib.smla_l1norm_run_tensors.restype = I32
    lib.smla_softmax_lse_run.argtypes = [P, ctypes.POINTER(_Tensors), P, P]
    lib.smla_softmax_lse_run.restype = I32
    lib.smla_l1norm_run_fused_lse.argtypes = [P, ctypes.POINTER(_Tensors), P, P]
    lib.smla_l1norm_run_fused_lse.restype = I32
    lib.smla_l1norm_io_sizes.argtypes = [P, ctypes.POINTER(IoSizes)]
    lib.smla_l1norm_io_sizes.restype = I32
    lib.smla_l1norm_run_from_host.argtypes = [P] + [P] * 6 + [P] * 6 + [P]
    lib.smla_l1norm_run_from_host.restype = I32
    lib.smla_l1norm_get_status.argtypes = [P, P, ctypes.POINTER(I32)]
    lib.smla_l1norm_get_status.restype = I32
    lib.smla_l1norm_schedule_host.argtypes = [ctypes.POINTER(_Desc), I32, I32, P, I64, P, ctypes.POINTER(PlanInfo)]
    lib.smla_l1norm_schedule_host.restype = I32
    lib.smla_status_string.argtypes = [I32]
    lib.smla_status_string.restype = ctypes.c_char_p
    lib.smla_get_last_cuda_error.argtypes = []
    lib.smla_get_last_cuda_error.restype = ctypes.c_char_p
    lib.smla_l1norm_run_noalloc.argtypes = [ctypes.POINTER(_Desc), P, P, P, P, P, P, P]
    lib.smla_l1norm_run_noalloc.restype = I32
    lib.smla_debug_gather.argtypes = [P, I32, I64, P, P, P, P, I64, P]
    lib.smla_debug_gather.restype = I32
    lib.smla_debug_noalloc_config.argtypes = [ctypes.POINTER(_Desc), I32, I32, ctypes.POINTER(PlanInfo)]
    lib.smla_debug_noalloc_config.restype = I32
    lib.smla_debug_wait_timeout_probe.argtypes = [I64, P, ctypes.POINTER(I32)]
    lib.smla_debug_wait_timeout_probe.restype = I32
    _ = F32
    _LIB = lib
    return lib


def _check(code: int, what: str):
    if code != SMLA_OK:
        detail = library().smla_get_last_cuda_error().decode() if code == SMLA_ERR_CUDA else ""
        raise SmlaError(code, what, detail)


def _i32_array(values):
    if values is None:
        return None, None
    vals = [int(v) for v in values]
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr, ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))


def _make_desc(*, layout="BSND", dtype="bf16", num_heads_q, num_heads_k=1, head_dim=512, batch_size=0,
               max_seqlen_q=0, max_seqlen_k=0, topk=0, mask_mode=0, cmp_ratio=1, softmax_scale=1.0,
               has_topk_length=False, cu_seqlens_q=None, cu_seqlens_k=None, topk_length_hint=None,
               num_ctas=0):
    keep = []
    d = _Desc()
    d.layout_q = d.layout_k = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    d.dtype = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    d.num_heads_q, d.num_heads_k, d.head_dim = num_heads_q, num_heads_k, head_dim
    d.batch_size, d.max_seqlen_q, d.max_seqlen_k = batch_size, max_seqlen_q, max_seqlen_k
    d.topk, d.mask_mode, d.cmp_ratio = topk, mask_mode, cmp_ratio
    d.softmax_scale = float(softmax_scale)
    d.has_topk_length = 1 if has_topk_length else 0
    for name, vals in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k),
                       ("topk_length_hint", topk_length_hint)):
        arr, ptr = _i32_array(None if vals is None else list(vals))
        if ptr is not None:
            setattr(d, name, ptr)
            keep.append(arr)
    d.num_ctas = num_ctas
    return d, keep


ITEM_FIELDS = 12


def schedule_host(num_ctas: int, want_items: bool = True, split_tiles: int = 0, **desc_kwargs):
    """Host-only scheduler view (no CUDA call): returns (items, cta_offsets, info)
    with items an (n, 12) int32 list-of-lists grouped by CTA.  ``split_tiles``:
    0 whole packs, n > 0 dense packs split into parts of n key tiles, -1 the
    dense L1-norm launch's own choice."""
    lib = library()
    d, keep = _make_desc(**desc_kwargs)
    info = PlanInfo()
    code = lib.smla_l1norm_schedule_host(ctypes.byref(d), num_ctas, split_tiles, None, 0, None, ctypes.byref(info))
    _check(code, "smla_l1norm_schedule_host")
    if not want_items:
        return None, None, info
    n = info.num_items
    items = (ctypes.c_int32 * (ITEM_FIELDS * max(1, n)))()
    offs = (ctypes.c_int32 * (num_ctas + 1))()
    code = lib.smla_l1norm_schedule_host(ctypes.byref(d), num_ctas, split_tiles, items, n, offs, ctypes.byref(info))
    _check(code, "smla_l1norm_schedule_host")
    rows = [list(items[ITEM_FIELDS * i: ITEM_FIELDS * i + ITEM_FIELDS]) for i in range(n)]
    del keep
    return rows, list(offs), info


def _ptr(t, name, required=True):
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """A validated operator description plus its device work schedule
    (``smla_l1norm_plan_create``).  Create once per shape; ``run`` per call."""

    def __init__(self, **desc_kwargs):
        self._lib = library()
        self.desc_kwargs = dict(desc_kwargs)
        d, keep = _make_desc(**desc_kwargs)
        h = ctypes.c_void_p()
        code = self._lib.smla_l1norm_plan_create(ctypes.byref(d), ctypes.byref(h))
        del keep
        _check(code, "smla_l1norm_plan_create")
        self._h = h

    @property
    def handle(self) -> int:
        return self._h.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.smla_l1norm_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def info(self) -> PlanInfo:
        info = PlanInfo()
        _check(self._lib.smla_l1norm_plan_get_info(self._h, ctypes.byref(info)), "plan_get_info")
        return info

    @property
    def output_shape(self) -> tuple:
        dims = (ctypes.c_int64 * 4)()
        nd = ctypes.c_int32()
        _check(self._lib.smla_l1norm_output_shape(self._h, dims, ctypes.byref(nd)), "output_shape")
        return tuple(dims[i] for i in range(nd.value))

    @property
    def io_sizes(self) -> IoSizes:
        s = IoSizes()
        _check(self._lib.smla_l1norm_io_sizes(self._h, ctypes.byref(s)), "io_sizes")
        return s

    def run(self, q, k, softmax_lse, sparse_indices=None, topk_length=None, out=None, stream=None,
            seqused_q=None, seqused_k=None, cmp_residual_k=None):
        """``smla_l1norm_run`` (``smla_l1norm_run_tensors`` when ``seqused_q``,
        ``seqused_k`` or ``cmp_residual_k`` is given: int32 CUDA tensors of one
        value per sequence); allocates ``out`` (fp32) if not given."""
        if out is None:
            import torch
            out = torch.empty(self.output_shape, dtype=torch.float32, device=q.device)
        if seqused_q is None and seqused_k is None and cmp_residual_k is None:
            code = self._lib.smla_l1norm_run(
                self._h, _ptr(q, "q"), _ptr(k, "k", required=False), _ptr(softmax_lse, "softmax_lse"),
                _ptr(sparse_indices, "sparse_indices", required=False),
                _ptr(topk_length, "topk_length", required=False), _ptr(out, "out"), _stream_handle(stream))
            _check(code, "smla_l1norm_run")
            return out
        t = _Tensors(_ptr(q, "q"), _ptr(k, "k", required=False), _ptr(softmax_lse, "softmax_lse"),
                     _ptr(sparse_indices, "sparse_indices", required=False),
                     _ptr(topk_length, "topk_length", required=False),
                     _ptr(seqused_q, "seqused_q", required=False),
                     _ptr(seqused_k, "seqused_k", required=False), _ptr(out, "out"),
                     _ptr(cmp_residual_k, "cmp_residual_k", required=False))
        code = self._lib.smla_l1norm_run_tensors(self._h, ctypes.byref(t), _stream_handle(stream))
        _check(code, "smla_l1norm_run_tensors")
        return out

    @property
    def lse_shape(self) -> tuple:
        """Shape of softmax_lse: (B, 1, S1, G) or (1, T1, G)."""
        d = self.desc_kwargs
        G = int(d["num_heads_q"]) // int(d.get("num_heads_k", 1))
        if d.get("layout", "BSND") == "TND":
            return (1, int(self.info.num_tokens), G)
        return (int(d.get("batch_size", 0)), 1, int(d.get("max_seqlen_q", 0)), G)

    def _tensors(self, q, k, sparse_indices, topk_length, seqused_q, seqused_k, out, cmp_residual_k=None):
        return _Tensors(_ptr(q, "q"), _ptr(k, "k", required=False), None,
                        _ptr(sparse_indices, "sparse_indices", required=False),
                        _ptr(topk_length, "topk_length", required=False),
                        _ptr(seqused_q, "seqused_q", required=False),
                        _ptr(seqused_k, "seqused_k", required=False), _ptr(out, "out", required=False),
                        _ptr(cmp_residual_k, "cmp_residual_k", required=False))

    def softmax_lse(self, q, k, sparse_indices=None, topk_length=None, lse_out=None, stream=None,
                    seqused_q=None, seqused_k=None, cmp_residual_k=None):
        """``smla_softmax_lse_run``: the forward LSE over the kept slots
        (natural log, fp32, -inf for a row with none); allocates ``lse_out``
        if not given."""
        if lse_out is None:
            import torch
            lse_out = torch.empty(self.lse_shape, dtype=torch.float32, device=q.device)
        t = self._tensors(q, k, sparse_indices, topk_length, seqused_q, seqused_k, None, cmp_residual_k)
        code = self._lib.smla_softmax_lse_run(self._h, ctypes.byref(t), _ptr(lse_out, "lse_out"),
                                              _stream_handle(stream))
        _check(code, "smla_softmax_lse_run")
        return lse_out

    def run_fused_lse(self, q, k, sparse_indices=None, topk_length=None, out=None, lse_out=None,
                      stream=None, seqused_q=None, seqused_k=None, cmp_residual_k=None):
        """``smla_l1norm_run_fused_lse``: the forward LSE and the operator
        from it in one launch; returns (out, lse_out)."""
        import torch
        if out is None:
            out = torch.empty(self.output_shape, dtype=torch.float32, device=q.device)
        if lse_out is None:
            lse_out = torch.empty(self.lse_shape, dtype=torch.float32, device=q.device)
        t = self._tensors(q, k, sparse_indices, topk_length, seqused_q, seqused_k, out, cmp_residual_k)
        code = self._lib.smla_l1norm_run_fused_lse(self._h, ctypes.byref(t), _ptr(lse_out, "lse_out"),
                                                   _stream_handle(stream))
        _check(code, "smla_l1norm_run_fused_lse")
        return out, lse_out

    def run_from_host(self, h, d, stream=None):
        """``smla_l1norm_run_from_host``: ``h`` and ``d`` map the roles
        q, k, lse, indices, topk_length, out to host (pinned) and device
        tensors (or None)."""
        roles = ("q", "k", "lse", "indices", "topk_length", "out")
        hp = [None if h.get(r) is None else h[r].data_ptr() for r in roles]
        dp = [None if d.get(r) is None else d[r].data_ptr() for r in roles]
        code = self._lib.smla_l1norm_run_from_host(self._h, *hp, *dp, _stream_handle(stream))
        _check(code, "smla_l1norm_run_from_host")

    def debug_gather(self, token, k, dump, sparse_indices=None, topk_length=None, mode=0, stream=None):
        """``smla_debug_gather``: the key producers alone for the work item of
        query ``token``; ``dump`` (a uint8 CUDA tensor) receives the ring
        stages as the tensor cores would read them."""
        code = self._lib.smla_debug_gather(self._h, int(mode), int(token), _ptr(k, "k", required=False),
                                           _ptr(sparse_indices, "sparse_indices", required=False),
                                           _ptr(topk_length, "topk_length", required=False),
                                           _ptr(dump, "dump"), int(dump.numel() * dump.element_size()),
                                           _stream_handle(stream))
        _check(code, "smla_debug_gather")
        return dump

    def status(self, stream=None):
        """(code, flags) from ``smla_l1norm_get_status`` (synchronises)."""
        flags = ctypes.c_int32()
        code = self._lib.smla_l1norm_get_status(self._h, _stream_handle(stream), ctypes.byref(flags))
        if code not in (SMLA_OK, SMLA_ERR_TIMEOUT, SMLA_WARN_BAD_INDEX):
            _check(code, "smla_l1norm_get_status")
        return code, flags.value


def wait_timeout_probe(timeout_ns: int = 50_000_000, stream=None):
    """Run a bounded device-side wait that nothing satisfies; returns (code, flags)."""
    lib = library()
    flags = ctypes.c_int32()
    code = lib.smla_debug_wait_timeout_probe(int(timeout_ns), _stream_handle(stream), ctypes.byref(flags))
    if code not in (SMLA_OK, SMLA_ERR_TIMEOUT):
        _check(code, "smla_debug_wait_timeout_probe")
    return code, flags.value


def run_noalloc(q, k, softmax_lse, out, sparse_indices=None, topk_length=None, stream=None,
                **desc_kwargs):
    """``smla_l1norm_run_noalloc``: the allocation-free entry point, for
    callers that cannot allocate device memory.  ``out`` must be given (this
    path allocates nothing); its scratch is a fixed device array shared by all
    calls on the device, so calls must not overlap on the GPU."""
    lib = library()
    d, keep = _make_desc(**desc_kwargs)
    code = lib.smla_l1norm_run_noalloc(
        ctypes.byref(d), _ptr(q, "q"), _ptr(k, "k", required=False), _ptr(softmax_lse, "softmax_lse"),
        _ptr(sparse_indices, "sparse_indices", required=False),
        _ptr(topk_length, "topk_length", required=False), _ptr(out, "out"), _stream_handle(stream))
    del keep
    _check(code, "smla_l1norm_run_noalloc")
    return out


def noalloc_config(num_sms: int, smem_optin: int, **desc_kwargs) -> PlanInfo:
    """``smla_debug_noalloc_config``: the launch shape ``run_noalloc`` would
    use on a device with ``num_sms`` SMs and ``smem_optin`` bytes of opt-in
    shared memory (host only, no CUDA call)."""
    lib = library()
    d, keep = _make_desc(**desc_kwargs)
    info = PlanInfo()
    code = lib.smla_debug_noalloc_config(ctypes.byref(d), int(num_sms), int(smem_optin), ctypes.byref(info))
    del keep
    _check(code, "smla_debug_noalloc_config")
    return info


_PLAN_CACHE = {}


def sparse_flash_mla_softmax_l1_norm(q, k, softmax_lse, *, sparse_indices=None, cu_seqlens_q=None,
                                     cu_seqlens_k=None, seqused_q=None, seqused_k=None,
                                     cmp_residual_k=None, topk_length=None, softmax_scale: float = 1.0,
                                     max_seqlen_k: int = 0, cmp_ratio: int = 1, mask_mode: int = 0,
                                     layout_q: str = "BSND", layout_k: str = "BSND",
                                     stream=None):
    """Functional form with the article's PyTorch argument names.  ``q``, ``k``,
    ``softmax_lse`` and the optional int32 tensors are CUDA tensors;
    ``cu_seqlens_q/k`` may be CUDA or CPU tensors or sequences (they are read
    on the host to build the schedule); ``seqused_q/k`` are int32 CUDA
    tensors, read on the device.  Plans are cached per shape."""
    import torch
    if layout_q != layout_k:
        raise ValueError("layout_q must equal layout_k")
    dtype = {torch.bfloat16: "bf16", torch.float16: "fp16"}.get(q.dtype)
    if dtype is None or k.dtype != q.dtype:
        raise ValueError("q and k must both be float16 or both bfloat16")
    cq = None if cu_seqlens_q is None else [int(x) for x in (cu_seqlens_q.tolist() if hasattr(cu_seqlens_q, "tolist") else cu_seqlens_q)]
    ck = None if cu_seqlens_k is None else [int(x) for x in (cu_seqlens_k.tolist() if hasattr(cu_seqlens_k, "tolist") else cu_seqlens_k)]
    topk = 0 if sparse_indices is None else int(sparse_indices.shape[-1])
    if layout_q == "TND":
        B = len(cq) - 1
        S1 = 0
        S2 = int(max_seqlen_k)
        N1 = int(q.shape[1])
    else:
        B, S1, N1 = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
        S2 = int(k.shape[1])
    key = (layout_q, dtype, N1, B, S1, S2, topk, mask_mode, cmp_ratio, float(softmax_scale),
           topk_length is not None, None if cq is None else tuple(cq), None if ck is None else tuple(ck),
           q.device.index)
    plan = _PLAN_CACHE.get(key)
    if plan is None:
        plan = Plan(layout=layout_q, dtype=dtype, num_heads_q=N1, batch_size=B, max_seqlen_q=S1,
                    max_seqlen_k=S2, topk=topk, mask_mode=mask_mode, cmp_ratio=cmp_ratio,
                    softmax_scale=softmax_scale, has_topk_length=topk_length is not None,
                    cu_seqlens_q=cq, cu_seqlens_k=ck)
        _PLAN_CACHE[key] = plan
    return plan.run(q, k, softmax_lse, sparse_indices=sparse_indices, topk_length=topk_length, stream=stream,
                    seqused_q=seqused_q, seqused_k=seqused_k, cmp_residual_k=cmp_residual_k)
