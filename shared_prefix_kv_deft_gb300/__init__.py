"""Python binding of the GB300 DeFT tree-attention decode library.

A thin ctypes layer over the C ABI in include/deft.h (libdeft.so, built by
`shared_prefix_kv_deft_gb300.build.build()`): the functions below have the
C names and only marshal arguments.  PyTorch provides device memory and the
current CUDA stream; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if libdeft.so is missing or a call
fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Tuple, Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libdeft.so")

DEFT_OUT_BF16 = 0
DEFT_OUT_F32 = 1

# deft_plan_array values (include/deft.h)
ARRAYS = {
    "chunk_seg_off": (0, np.int32), "chunk_q_off": (1, np.int32), "chunk_q": (2, np.int32),
    "seg_node": (3, np.int32), "seg_tok_begin": (4, np.int32), "seg_tok_len": (5, np.int32),
    "seg_mask": (6, np.uint64), "chunk_mask": (7, np.uint64), "q_slot_off": (8, np.int32),
    "q_slot": (9, np.int32), "node_cover": (10, np.uint64), "node_order": (11, np.int32),
    "fma_items": (12, np.int32), "mma_items": (13, np.int32), "fallback_items": (14, np.int32),
    "naive_chunk_seg_off": (15, np.int32), "naive_chunk_q": (16, np.int32),
    "naive_seg_node": (17, np.int32), "naive_seg_tok_begin": (18, np.int32),
    "naive_seg_tok_len": (19, np.int32), "naive_q_slot_off": (20, np.int32),
    "naive_q_slot": (21, np.int32), "fma_direct": (22, np.uint32),
    "fallback_direct": (23, np.uint32), "merge_q": (24, np.int32),
}

# Symbols the header declares (checked by the tests).
EXPORTS = ["deft_plan", "deft_plan_at", "deft_plan_ex", "deft_plan_rebuild", "deft_plan_stats_get",
           "deft_plan_get", "deft_plan_upload", "deft_workspace_bytes", "deft_tree_attn",
           "deft_naive_attn", "deft_tree_attn_ex", "deft_step_status", "deft_check_pages",
           "deft_plan_update", "deft_pages_create", "deft_pages_free", "deft_pages_alloc",
           "deft_pages_retain", "deft_pages_release", "deft_pages_free_count", "deft_pages_refcount",
           "deft_plan_free", "deft_status_str", "deft_version", "deft_trace_enable",
           "deft_trace_read", "deft_tree_attn_noalloc", "deft_tree_attn_host"]

KERNEL_NAMES = {0: "phase1_fma", 1: "phase1_mma", 2: "phase2_merge"}
PLAN_TREE_ONLY = 1   # deft_plan_ex flags
PLAN_TENSOR_PACK = 2
# deft_tree_attn_ex flags
STEP_NAIVE = 1
STEP_CUDA_CORES = 2
STEP_SEPARATE_MERGE = 4


class DeftError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({status_str(status)})")
        self.status = status


class TraceRecord(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("family", ctypes.c_int32),
                ("bucket", ctypes.c_int32), ("fallback", ctypes.c_int32),
                ("items", ctypes.c_int32), ("ms", ctypes.c_float)]


class PlanStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_nodes", "num_queries", "gqa_group", "chunk_target", "mask_words", "num_chunks",
        "num_segments", "num_slots", "num_fma_items", "num_mma_items", "num_fallback_items",
        "max_chunk_tokens", "max_slots_per_query", "naive_num_chunks", "naive_num_slots",
        "naive_num_segments", "num_merge_queries", "reserved0")] + [(n, ctypes.c_int64) for n in (
        "unique_tokens", "naive_tokens", "planned_tokens", "pair_tokens", "device_bytes")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None


def load(path: str = LIB_PATH):
    """Load libdeft.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "shared_prefix_kv_deft_gb300.build.build() (no fallback exists)")
    lib = ctypes.CDLL(path)
    P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    lib.deft_plan.argtypes = [P, P, i32, P, i32, i32, i32, ctypes.POINTER(P)]
    lib.deft_plan_at.argtypes = [P, P, i32, P, P, i32, i32, i32, ctypes.POINTER(P)]
    lib.deft_plan_ex.argtypes = [P, P, i32, P, P, i32, i32, i32, i32, ctypes.POINTER(P)]
    lib.deft_plan_rebuild.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32]
    lib.deft_plan_stats_get.argtypes = [P, ctypes.POINTER(PlanStats)]
    lib.deft_plan_get.argtypes = [P, i32, P, sz]
    lib.deft_plan_upload.argtypes = [P, P]
    lib.deft_workspace_bytes.argtypes = [P, i32, i32]
    lib.deft_workspace_bytes.restype = sz
    attn = [P, P, P, P, P, i32, i32, i32, i32, i32, f32, P, P, i32, P, P, sz, P]
    lib.deft_tree_attn.argtypes = attn
    lib.deft_naive_attn.argtypes = attn
    lib.deft_tree_attn_ex.argtypes = attn[:-1] + [i32, P]
    lib.deft_tree_attn_host.argtypes = [P] + attn[:-1] + [P, P, P]
    lib.deft_step_status.argtypes = [P, P, ctypes.POINTER(i32)]
    lib.deft_check_pages.argtypes = [P, i32, P, P, ctypes.c_int64, i32, i32]
    lib.deft_plan_update.argtypes = [P, P, i32]
    lib.deft_pages_create.argtypes = [i32, ctypes.POINTER(P)]
    lib.deft_pages_free.argtypes = [P]
    lib.deft_pages_free.restype = None
    for fn in ("deft_pages_alloc", "deft_pages_retain", "deft_pages_release"):
        getattr(lib, fn).argtypes = [P, i32, P]
    lib.deft_pages_free_count.argtypes = [P]
    lib.deft_pages_refcount.argtypes = [P, i32]
    lib.deft_tree_attn_noalloc.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f32, P, P,
                                           i32, P, P]
    lib.deft_plan_free.argtypes = [P]
    lib.deft_plan_free.restype = None
    lib.deft_status_str.argtypes = [ctypes.c_int]
    lib.deft_status_str.restype = ctypes.c_char_p
    lib.deft_version.argtypes = []
    lib.deft_trace_enable.argtypes = [i32]
    lib.deft_trace_read.argtypes = [ctypes.POINTER(TraceRecord), i32, ctypes.POINTER(i32)]
    for fn in ("deft_plan", "deft_plan_at", "deft_plan_ex", "deft_plan_rebuild", "deft_plan_stats_get",
               "deft_plan_get", "deft_plan_upload", "deft_tree_attn", "deft_naive_attn", "deft_version",
               "deft_trace_enable", "deft_trace_read", "deft_tree_attn_noalloc", "deft_tree_attn_ex",
               "deft_step_status", "deft_check_pages", "deft_plan_update", "deft_pages_create",
               "deft_pages_alloc", "deft_pages_retain", "deft_pages_release", "deft_pages_free_count",
               "deft_pages_refcount"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load().deft_status_str(int(status)).decode()


def _check(fn: str, rc: int):
    if rc != 0:
        raise DeftError(fn, rc)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _plan_flags(naive: bool, tensor_pack: bool) -> int:
    return (0 if naive else PLAN_TREE_ONLY) | (PLAN_TENSOR_PACK if tensor_pack else 0)


def _ptr(a: np.ndarray) -> int:
    # The address as an int (ctypes converts it for c_void_p parameters);
    # cheaper than building a ctypes pointer object.
    return a.ctypes.data


class Plan:
    """Owner of a deft_plan_t handle (deft_plan_ex ... deft_plan_free).
    query_pos: per query, the token of its node it sits at (-1: the last);
    None: every query at its node's last token.  naive=False: tree-only plan
    (DEFT_PLAN_TREE_ONLY; deft_naive_attn refuses it)."""

    def __init__(self, parent, node_len, query_node, chunk_target: int = 256, gqa_group: int = 1,
                 query_pos=None, naive: bool = True, tensor_pack: bool = False):
        lib = load()
        par, ln, qn = _i32(parent), _i32(node_len), _i32(query_node)
        pos = None if query_pos is None else _i32(query_pos)
        h = ctypes.c_void_p()
        _check("deft_plan_ex", lib.deft_plan_ex(_ptr(par), _ptr(ln), int(par.shape[0]), _ptr(qn),
                                                None if pos is None else _ptr(pos), int(qn.shape[0]),
                                                int(chunk_target), int(gqa_group),
                                                _plan_flags(naive, tensor_pack), ctypes.byref(h)))
        self.handle = h
        self._stats = None
        self._staged = {}

    def _stage(self, slot: int, a) -> Tuple[int, int]:
        """a copied into this plan's int32 staging buffer `slot` (kept across
        rebuilds, its address taken once): (length, address).  The library
        copies the inputs it keeps, so the buffers are only read during the
        call."""
        a = np.asarray(a)
        n = int(a.shape[0])
        buf, addr = self._staged.get(slot, (None, 0))
        if buf is None or buf.shape[0] < n:
            buf = np.empty(max(2 * n, 64), dtype=np.int32)
            addr = buf.ctypes.data
            self._staged[slot] = (buf, addr)
        buf[:n] = a
        return n, addr

    @property
    def stats(self) -> dict:
        """deft_plan_stats_get, read once per build."""
        if self._stats is None:
            st = PlanStats()
            _check("deft_plan_stats_get", load().deft_plan_stats_get(self.handle, ctypes.byref(st)))
            self._stats = st.as_dict()
        return self._stats

    def rebuild(self, parent, node_len, query_node, chunk_target: int = 256, gqa_group: int = 1,
                query_pos=None, naive: bool = True, tensor_pack: bool = False):
        """deft_plan_rebuild: plan a new tree into this plan, keeping its device
        allocation and staging buffer; upload() again before the next step.
        On error (DeftError) the plan is unchanged."""
        n, par = self._stage(0, parent)
        n_len, ln = self._stage(1, node_len)
        nq, qn = self._stage(2, query_node)
        pos = None if query_pos is None else self._stage(3, query_pos)[1]
        if n_len != n:
            raise ValueError("parent and node_len differ in length")
        _check("deft_plan_rebuild", load().deft_plan_rebuild(
            self.handle, par, ln, n, qn, pos, nq, int(chunk_target), int(gqa_group),
            _plan_flags(naive, tensor_pack)))
        self._stats = None

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.deft_plan_free(h)
            self.handle = None

    def _count(self, name: str) -> int:
        s = self.stats
        W, C, S = s["mask_words"], s["num_chunks"], s["num_segments"]
        counts = {
            "chunk_seg_off": C + 1, "chunk_q_off": C + 1, "chunk_q": s["num_slots"],
            "seg_node": S, "seg_tok_begin": S, "seg_tok_len": S, "seg_mask": S * W,
            "chunk_mask": C * W, "q_slot_off": s["num_queries"] + 1, "q_slot": s["num_slots"],
            "node_cover": s["num_nodes"] * W, "node_order": s["num_nodes"],
            "fma_items": 3 * s["num_fma_items"], "mma_items": 3 * s["num_mma_items"],
            "fallback_items": 3 * s["num_fallback_items"],
            "naive_chunk_seg_off": s["naive_num_chunks"] + 1,
            "naive_chunk_q": s["naive_num_slots"], "naive_seg_node": s["naive_num_segments"],
            "naive_seg_tok_begin": s["naive_num_segments"],
            "naive_seg_tok_len": s["naive_num_segments"],
            "naive_q_slot_off": s["num_queries"] + 1, "naive_q_slot": s["naive_num_slots"],
            "fma_direct": s["num_fma_items"], "fallback_direct": s["num_fallback_items"],
            "merge_q": s["num_merge_queries"],
        }
        return counts[name]

    def get(self, name: str) -> np.ndarray:
        """Host copy of one plan array (deft_plan_get)."""
        which, dt = ARRAYS[name]
        out = np.zeros(max(self._count(name), 1), dtype=dt)
        _check("deft_plan_get", load().deft_plan_get(self.handle, which, _ptr(out), out.nbytes))
        return out[: self._count(name)]

    def upload(self, stream=None):
        _check("deft_plan_upload", load().deft_plan_upload(self.handle, _stream(stream)))

    def workspace_bytes(self, num_q_heads: int, head_dim: int) -> int:
        return int(load().deft_workspace_bytes(self.handle, int(num_q_heads), int(head_dim)))

    def update(self, node_len):
        """deft_plan_update: the same tree with new node lengths (tokens
        appended, pruned subtrees at 0); upload() again before the next step."""
        n, ln = self._stage(1, node_len)
        _check("deft_plan_update", load().deft_plan_update(self.handle, ln, n))
        self._stats = None

    def step_status(self, stream=None) -> int:
        """deft_step_status: 0, or the code of a kernel wait that ran out in an
        earlier step (the codes are cleared by the call)."""
        code = ctypes.c_int32()
        rc = load().deft_step_status(self.handle, _stream(stream), ctypes.byref(code))
        if rc not in (0, -9):
            _check("deft_step_status", rc)
        return int(code.value)


def _stream(stream):
    """The raw cudaStream_t (an int) of `stream`, or of torch's current
    stream when it is None."""
    if stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            # The current stream's handle without building a Stream object
            # (~0.3 us against ~3 us for torch.cuda.current_stream()).
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclass
class StepBuffers:
    out: "object"
    lse: "object"
    workspace: "object"


def alloc_buffers(plan: Plan, num_queries: int, num_q_heads: int, head_dim: int, device="cuda",
                  out_dtype: int = DEFT_OUT_BF16) -> StepBuffers:
    """Device output, lse and workspace tensors for one step (torch memory)."""
    import torch
    odt = torch.bfloat16 if out_dtype == DEFT_OUT_BF16 else torch.float32
    ws = plan.workspace_bytes(num_q_heads, head_dim)
    return StepBuffers(torch.empty((num_queries, num_q_heads, head_dim), dtype=odt, device=device),
                       torch.empty((num_queries, num_q_heads), dtype=torch.float32, device=device),
                       torch.empty(ws, dtype=torch.uint8, device=device))


def _attn(fn_name: str, q, k_pages, v_pages, node_page_off, page_id, plan: Plan,
          bufs: Optional[StepBuffers] = None, scale: Optional[float] = None,
          out_dtype: int = DEFT_OUT_BF16, stream=None, flags: int = 0):
    import torch
    lib = load()
    Q, Hq, d = q.shape
    Hkv, P = k_pages.shape[1], k_pages.shape[2]
    if bufs is None:
        bufs = alloc_buffers(plan, Q, Hq, d, q.device, out_dtype)
    for t in (q, k_pages, v_pages):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k_pages and v_pages must be contiguous bf16 CUDA tensors")
    for t in (node_page_off, page_id):
        if t.dtype != torch.int32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("node_page_off and page_id must be contiguous int32 CUDA tensors")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    odt = DEFT_OUT_BF16 if bufs.out.dtype == torch.bfloat16 else DEFT_OUT_F32
    args = [q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), node_page_off.data_ptr(),
            page_id.data_ptr(), int(k_pages.shape[0]), int(Hq), int(Hkv), int(d),
            int(P), float(scale), plan.handle, bufs.out.data_ptr(), odt,
            bufs.lse.data_ptr(), bufs.workspace.data_ptr(), int(bufs.workspace.numel())]
    if fn_name == "deft_tree_attn_ex":
        args.append(int(flags))
    rc = getattr(lib, fn_name)(*args, _stream(stream))
    _check(fn_name, rc)
    return bufs.out, bufs.lse


def deft_tree_attn(q, k_pages, v_pages, node_page_off, page_id, plan: Plan, bufs=None,
                   scale=None, out_dtype=DEFT_OUT_BF16, stream=None, flags: int = 0):
    """One DeFT tree-attention step; returns (out, lse) device tensors.
    flags (STEP_*): deft_tree_attn_ex's options; 0 calls deft_tree_attn."""
    return _attn("deft_tree_attn_ex" if flags else "deft_tree_attn", q, k_pages, v_pages,
                 node_page_off, page_id, plan, bufs, scale, out_dtype, stream, flags)


def _host_step_args(q_host, q, k_pages, v_pages, node_page_off, page_id, plan: Plan, bufs: StepBuffers,
                    out_host, lse_host, scale):
    """The checked arguments of deft_tree_attn_host, the stream left out."""
    import torch
    Q, Hq, d = q.shape
    Hkv, P = k_pages.shape[1], k_pages.shape[2]
    for t in (q, k_pages, v_pages):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k_pages and v_pages must be contiguous bf16 CUDA tensors")
    if q_host.dtype != torch.bfloat16 or not q_host.is_contiguous() or q_host.is_cuda or q_host.shape != q.shape:
        raise ValueError("q_host must be a contiguous bf16 host tensor shaped like q")
    for h, dv in ((out_host, bufs.out), (lse_host, bufs.lse)):
        if h.is_cuda or not h.is_contiguous() or h.dtype != dv.dtype or h.shape != dv.shape:
            raise ValueError("out_host / lse_host must be contiguous host tensors shaped like the outputs")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    odt = DEFT_OUT_BF16 if bufs.out.dtype == torch.bfloat16 else DEFT_OUT_F32
    return (q_host.data_ptr(), q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), node_page_off.data_ptr(),
            page_id.data_ptr(), int(k_pages.shape[0]), int(Hq), int(Hkv), int(d), int(P), float(scale), plan.handle,
            bufs.out.data_ptr(), odt, bufs.lse.data_ptr(), bufs.workspace.data_ptr(), int(bufs.workspace.numel()),
            out_host.data_ptr(), lse_host.data_ptr())


def deft_tree_attn_host(q_host, q, k_pages, v_pages, node_page_off, page_id, plan: Plan, bufs: StepBuffers,
                        out_host, lse_host, scale=None, stream=None):
    """deft_tree_attn_host: q_host (host, pinned for an asynchronous copy) is
    copied into the device buffer q, the step runs, and out / lse are copied
    into out_host / lse_host, all on the stream; synchronise it before
    reading the host outputs."""
    args = _host_step_args(q_host, q, k_pages, v_pages, node_page_off, page_id, plan, bufs, out_host, lse_host,
                           scale)
    _check("deft_tree_attn_host", load().deft_tree_attn_host(*args, _stream(stream)))
    return out_host, lse_host


class HostStep:
    """deft_tree_attn_host bound to one set of buffers, for a decode loop
    that runs the same shapes every step: the arguments are checked and
    marshalled once, each call is one library call on the stream.  The
    object holds the tensors and the plan, so their addresses stay valid;
    refill q_host (and rebuild or update the plan, then upload it) between
    calls, and synchronise the stream before reading out_host / lse_host."""

    def __init__(self, q_host, q, k_pages, v_pages, node_page_off, page_id, plan: Plan, bufs: StepBuffers,
                 out_host, lse_host, scale=None):
        self._args = _host_step_args(q_host, q, k_pages, v_pages, node_page_off, page_id, plan, bufs, out_host,
                                     lse_host, scale)
        self._held = (q_host, q, k_pages, v_pages, node_page_off, page_id, plan, bufs, out_host, lse_host)
        self._fn = load().deft_tree_attn_host
        self.out_host, self.lse_host = out_host, lse_host

    def __call__(self, stream=None):
        rc = self._fn(*self._args, _stream(stream))
        if rc:
            _check("deft_tree_attn_host", rc)
        return self.out_host, self.lse_host


def deft_naive_attn(q, k_pages, v_pages, node_page_off, page_id, plan: Plan, bufs=None,
                    scale=None, out_dtype=DEFT_OUT_BF16, stream=None):
    """The per-query flash-decoding form of the same step (IO comparison)."""
    return _attn("deft_naive_attn", q, k_pages, v_pages, node_page_off, page_id, plan, bufs,
                 scale, out_dtype, stream)


def deft_plan(parent, node_len, query_node, chunk_target: int = 256, gqa_group: int = 1,
              query_pos=None, naive: bool = True, tensor_pack: bool = False) -> Plan:
    return Plan(parent, node_len, query_node, chunk_target, gqa_group, query_pos, naive, tensor_pack)


class PagePool:
    """deft_pages_*: a host pool of KV page numbers with reference counts."""

    def __init__(self, num_pages: int):
        h = ctypes.c_void_p()
        _check("deft_pages_create", load().deft_pages_create(int(num_pages), ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.deft_pages_free(h)
            self.handle = None

    def alloc(self, n: int) -> np.ndarray:
        out = np.zeros(max(int(n), 1), dtype=np.int32)
        _check("deft_pages_alloc", load().deft_pages_alloc(self.handle, int(n), _ptr(out)))
        return out[: int(n)]

    def retain(self, ids):
        ids = _i32(ids)
        _check("deft_pages_retain", load().deft_pages_retain(self.handle, int(ids.size),
                                                             _ptr(ids) if ids.size else None))

    def release(self, ids):
        ids = _i32(ids)
        _check("deft_pages_release", load().deft_pages_release(self.handle, int(ids.size),
                                                               _ptr(ids) if ids.size else None))

    @property
    def free_count(self) -> int:
        return int(load().deft_pages_free_count(self.handle))

    def refcount(self, page: int) -> int:
        return int(load().deft_pages_refcount(self.handle, int(page)))


def deft_check_pages(node_len, node_page_off, page_id, num_pages: int, page_size: int = 16) -> int:
    """deft_check_pages on host arrays: 0 (DEFT_OK) or the status code."""
    ln, npo, pid = _i32(node_len), _i32(node_page_off), _i32(page_id)
    return int(load().deft_check_pages(_ptr(ln), int(ln.shape[0]), _ptr(npo),
                                       _ptr(pid) if pid.size else None, int(pid.size),
                                       int(num_pages), int(page_size)))


def trace_enable(on: bool = True):
    _check("deft_trace_enable", load().deft_trace_enable(1 if on else 0))


def trace_read(cap: int = 1 << 16):
    """Per-launch records since the last read: list of dicts (waits for the events)."""
    recs = (TraceRecord * cap)()
    n = ctypes.c_int32()
    _check("deft_trace_read", load().deft_trace_read(recs, cap, ctypes.byref(n)))
    return [{"kernel": KERNEL_NAMES.get(r.kernel, str(r.kernel)), "family": r.family,
             "bucket": r.bucket, "fallback": r.fallback, "items": r.items, "ms": r.ms}
            for r in recs[: n.value]]


def version() -> int:
    return int(load().deft_version())
