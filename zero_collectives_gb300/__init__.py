"""Python binding of libdpred (argument marshalling only).

Every function here forwards to the C-ABI entry point of the same name in
``libdpred.so`` (declared in ``include/dpred.h``); all device work runs in that
library's CUDA kernels.  There is no fallback: if the library is missing or a
call fails, a ``DpredError`` is raised.  PyTorch is used only for device
memory and streams.
"""
from __future__ import annotations

import ctypes
import weakref
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# DPRED_CHECKED=1 in the environment loads the checked build instead (every
# flush-kernel access bounds-tested on the device; build it with
# zero_collectives_gb300.build.build(checked=True)).
CHECKED = os.environ.get("DPRED_CHECKED", "0") == "1"
LIB_PATH = os.path.join(_HERE, "libdpred_checked.so" if CHECKED else "libdpred.so")

BF16, F32 = 0, 1
MAX_WORLD = 64
DTYPE_NAMES = {BF16: "BFloat16", F32: "Float"}  # names the probe line prints

# dpred_task: {int32 param_id, int32 reserved, int64 offset, int64 numel}
TASK_DTYPE = np.dtype([("param_id", "<i4"), ("pad", "<i4"), ("offset", "<i8"), ("numel", "<i8")])

E_CODES = {-1: "DPRED_E_INVAL", -2: "DPRED_E_ALIGN", -3: "DPRED_E_SIZE", -4: "DPRED_E_MISMATCH",
           -5: "DPRED_E_CUDA", -6: "DPRED_E_TIMEOUT", -7: "DPRED_E_BOUNDS"}


class DpredError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{E_CODES.get(code, code)}: {msg}")
        self.code = code


class _Group(ctypes.Structure):
    _fields_ = [("comm_size", ctypes.c_int32), ("n_params", ctypes.c_int32),
                ("comm_ranks", ctypes.c_void_p), ("numel", ctypes.c_void_p)]


class _Probe(ctypes.Structure):
    _fields_ = [("flush_index", ctypes.c_int64), ("tasks", ctypes.c_int64), ("reduced_elems", ctypes.c_int64),
                ("owner_tasks", ctypes.c_int64), ("owner_elems", ctypes.c_int64),
                ("kept_elems", ctypes.c_int64 * MAX_WORLD)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libdpred.so; raises ImportError when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            how = "build.build(checked=True)" if CHECKED else "__graft_entry__.build()"
            raise ImportError(f"{LIB_PATH} is missing: build it with {how} (there is no fallback path)")
        L = ctypes.CDLL(LIB_PATH)
        i32, i64, vp, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
        L.dpred_last_error.restype = ctypes.c_char_p
        L.dpred_version.restype = ctypes.c_char_p
        L.dpred_build_owner_map.argtypes = [i32, i32, vp, i32, i32, vp, vp, vp, vp, vp]
        L.dpred_owner_map_digest.restype = ctypes.c_uint64
        L.dpred_owner_map_digest.argtypes = [i32, vp, vp, vp]
        L.dpred_build_owner_map_device.argtypes = [i32, i32, vp, i32, vp, i32, vp, vp, vp, vp, vp]
        L.dpred_flush_probe.argtypes = [i32, vp, i32, vp, i32, vp, i32, vp]
        L.dpred_probe_format.argtypes = [vp, i32, i32, i32, i32, ctypes.c_char_p, ctypes.c_size_t]
        L.dpred_flush_workspace_bytes.restype = ctypes.c_size_t
        L.dpred_flush_workspace_bytes.argtypes = [i32, i32]
        L.dpred_flush_bucket.argtypes = [i32, i32, vp, i64, vp, i32, vp, i32, i32, vp, i32, i32, i32, vp, vp,
                                         ctypes.c_size_t, vp]
        L.dpred_executor_create.argtypes = [i32, i32, i32, i32, i32, vp, i32, vp, i64, i32, vp, vp, vp, vp, vp,
                                            ctypes.c_size_t, vp]
        L.dpred_executor_flush.argtypes = [vp, i32, vp, vp]
        L.dpred_executor_flush_all.argtypes = [vp, vp, vp]
        L.dpred_executor_set_overlap.argtypes = [vp, i32]
        L.dpred_executor_create_partitioned.argtypes = [i32, i32, i32, i32, vp, i64, i32, vp, vp, vp, vp, i32, i64,
                                                        vp, vp, ctypes.c_size_t, vp]
        L.dpred_executor_overlap_eligible.argtypes = [vp]
        L.dpred_executor_flush_all_from_host.argtypes = [vp, vp, i64, i32, vp, vp, vp, vp, vp]
        L.dpred_executor_destroy.argtypes = [vp]
        L.dpred_flush_bucket_noalloc.argtypes = [i32, i32, vp, i64, vp, i32, vp, i32, i32, vp, i32, i32, i32, vp,
                                                 vp]
        L.dpred_accumulate_microbatch.argtypes = [i32, i64, vp, i32, vp, i32, i32, f32, vp, vp]
        L.dpred_flush_bucket_partitioned.argtypes = [i32, i32, vp, i64, vp, i32, vp, i32, i64, i32, vp, i32, vp, vp,
                                                     ctypes.c_size_t, vp]
        L.dpred_bucket_relayout_workspace_bytes.restype = ctypes.c_size_t
        L.dpred_bucket_relayout_workspace_bytes.argtypes = [i32, i32]
        L.dpred_bucket_relayout.argtypes = [i32, i32, vp, i64, vp, i32, vp, i32, i64, i64, vp, i64, vp, vp,
                                            ctypes.c_size_t, vp]
        L.dpred_allgather_schedule_steps.argtypes = [i32, i32]
        L.dpred_allgather_schedule_init.argtypes = [i32, i32, i64, i32, vp, vp, vp]
        L.dpred_allgather_schedule_step.argtypes = [i32, i32, i64, i32, vp, i32, vp]
        L.dpred_accumulator_save.argtypes = [i32, i64, vp, vp, vp]
        L.dpred_accumulator_restore.argtypes = [i32, i64, vp, vp, vp]
        L.dpred_reduce_scatter.argtypes = [i32, i64, i32, vp, i32, vp, i32, vp]
        L.dpred_allgather.argtypes = [i32, i64, i32, vp, vp, i32, vp]
        L.dpred_device_status.argtypes = [vp, i32]
        L.dpred_set_flush_path.argtypes = [i32]
        L.dpred_set_allgather_form.argtypes = [i32]
        L.dpred_fill_pattern.argtypes = [vp, ctypes.c_size_t, ctypes.c_uint32, i32, i32, vp]
        L.dpred_stream_mixed.argtypes = [vp, ctypes.c_size_t, vp, ctypes.c_size_t, vp]
        L.dpred_selftest_wait_timeout.argtypes = [i64, vp]
        L.dpred_selftest_bounds.argtypes = [vp]
        L.dpred_selftest_prediv.argtypes = [i32, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint32)]
        L.dpred_host_mapped_pointer.argtypes = [vp, ctypes.POINTER(vp)]
        L.dpred_executor_flush_all_mapped.argtypes = L.dpred_executor_flush_all_from_host.argtypes
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise DpredError(rc, lib().dpred_last_error().decode())


def _dtype_code(t) -> int:
    import torch
    dt = t.dtype
    if dt is torch.bfloat16:
        return BF16
    if dt is torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _stream(stream) -> int:
    import torch
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:  # the current stream's handle without building a Stream object
            return raw(torch._C._cuda_getDevice())
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_PTRS: dict = {}


def _ptr(a: np.ndarray) -> int:
    """Address of a numpy array's data, remembered per live array (numpy's
    own .ctypes.data costs microseconds per call).  An entry is used only
    while the same array object, with the same size, is alive."""
    e = _PTRS.get(id(a))
    if e is not None and e[0]() is a and e[1] == a.size:
        return e[2]
    if len(_PTRS) > 4096:
        _PTRS.clear()
    v = a.ctypes.data
    _PTRS[id(a)] = (weakref.ref(a), a.size, v)
    return v


def version() -> str:
    return lib().dpred_version().decode()


# -------------------------------------------------------------- owner map ---

@dataclass
class OwnerMap:
    owner: np.ndarray      # int32 per parameter, -1 = AllReduce
    holder_lo: np.ndarray  # int32
    holder_hi: np.ndarray  # int32
    n_owned: int
    n_total: int

    def digest(self) -> int:
        """64-bit digest of the map (dpred_owner_map_digest), for cross-rank checks."""
        n = len(self.owner)
        return int(lib().dpred_owner_map_digest(n, self.owner.ctypes.data, self.holder_lo.ctypes.data,
                                                self.holder_hi.ctypes.data))

    def report(self) -> str:
        """The init-time ratio report of the DeepSpeed issue (section "Additional context")."""
        return f"DeepCompile reduce_to_owner: {self.n_owned}/{self.n_total} gradients reduce to one rank"


def build_owner_map(world: int, groups, reduce_to_owner: bool = True, rank: int = 0) -> OwnerMap:
    """groups: list of (comm_ranks or None, numel sequence) in group order."""
    keep = []
    arr = (_Group * max(len(groups), 1))()
    total = 0
    for i, (ranks, numel) in enumerate(groups):
        n = np.ascontiguousarray(numel, dtype=np.int64)
        keep.append(n)
        arr[i].n_params = len(n)
        arr[i].numel = n.ctypes.data if len(n) else None
        if ranks is None:
            arr[i].comm_size = world
            arr[i].comm_ranks = None
        else:
            r = np.ascontiguousarray(ranks, dtype=np.int32)
            keep.append(r)
            arr[i].comm_size = len(r)
            arr[i].comm_ranks = r.ctypes.data
        total += len(n)
    owner = np.empty(total, np.int32)
    lo = np.empty(total, np.int32)
    hi = np.empty(total, np.int32)
    n_owned, n_total = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().dpred_build_owner_map(world, rank, arr, len(groups), int(reduce_to_owner), owner.ctypes.data,
                                       lo.ctypes.data, hi.ctypes.data, ctypes.byref(n_owned), ctypes.byref(n_total)))
    return OwnerMap(owner, lo, hi, n_owned.value, n_total.value)


def build_owner_map_device(world: int, numel, comm_ranks=None, reduce_to_owner: bool = True, stream=None):
    """Owner map of one group on the device.  numel: CUDA int64 tensor;
    comm_ranks: CUDA int32 tensor or None.  Returns CUDA int32 tensors
    (owner, holder_lo, holder_hi, counts[n_owned, n_total])."""
    import torch
    if numel.dtype != torch.int64 or not numel.is_cuda or not numel.is_contiguous():
        raise ValueError("numel must be a contiguous CUDA int64 tensor")
    n = numel.numel()
    dev = numel.device
    owner = torch.empty(n, dtype=torch.int32, device=dev)
    lo = torch.empty(n, dtype=torch.int32, device=dev)
    hi = torch.empty(n, dtype=torch.int32, device=dev)
    counts = torch.empty(2, dtype=torch.int32, device=dev)
    cs = world if comm_ranks is None else comm_ranks.numel()
    _check(lib().dpred_build_owner_map_device(world, n, numel.data_ptr(), cs,
                                              None if comm_ranks is None else comm_ranks.data_ptr(),
                                              int(reduce_to_owner), owner.data_ptr(), lo.data_ptr(), hi.data_ptr(),
                                              counts.data_ptr(), _stream(stream)))
    return owner, lo, hi, counts


# ------------------------------------------------------------------ probe ---

@dataclass
class Probe:
    flush_index: int
    tasks: int
    reduced_elems: int
    owner_tasks: int
    owner_elems: int
    kept_elems: list

    def line(self, rank: int, dtype: int, pre_div: bool) -> str:
        """The probe line of the DeepSpeed issue ("reduce_probe"), for one rank,
        as dpred_probe_format writes it."""
        p = _Probe()
        p.flush_index, p.tasks, p.reduced_elems = self.flush_index, self.tasks, self.reduced_elems
        p.owner_tasks, p.owner_elems = self.owner_tasks, self.owner_elems
        for r, k in enumerate(self.kept_elems):
            p.kept_elems[r] = k
        buf = ctypes.create_string_buffer(256)
        _check(lib().dpred_probe_format(ctypes.byref(p), len(self.kept_elems), int(rank), int(dtype),
                                        1 if pre_div else 0, buf, len(buf)))
        return buf.value.decode()


class ProbeLog:
    """Prints one probe line per flush for the first ``limit`` flushes (the
    issue's reduce_probe prints the first 20)."""

    def __init__(self, rank: int = 0, limit: int = 20, sink=print):
        self.rank, self.limit, self.sink, self.count = rank, limit, sink, 0

    def next_index(self) -> int:
        return self.count

    def record(self, probe: Probe, dtype: int, pre_div: bool) -> None:
        if probe.flush_index < self.limit:
            self.sink(probe.line(self.rank, dtype, pre_div))
        self.count += 1


def _probe_from(p: _Probe, world: int) -> Probe:
    return Probe(p.flush_index, p.tasks, p.reduced_elems, p.owner_tasks, p.owner_elems, p.kept_elems[:world])


def _tasks_arg(tasks: np.ndarray) -> np.ndarray:
    if type(tasks) is np.ndarray and tasks.dtype is TASK_DTYPE and tasks.flags.c_contiguous:
        return tasks
    t = np.ascontiguousarray(tasks)
    if t.dtype != TASK_DTYPE:
        t = np.ascontiguousarray(t.astype(TASK_DTYPE))
    return t


def _owner_arg(owner):
    if owner is None:
        return None
    if type(owner) is np.ndarray and owner.dtype == np.int32 and owner.flags.c_contiguous:
        return owner
    return np.ascontiguousarray(owner, dtype=np.int32)


class DstTable:
    """Host array [world * n_tasks] of destination device pointers (0 = empty
    buffer), built once and reused across flushes."""

    def __init__(self, world: int, n_tasks: int, ptrs):
        ptrs = list(ptrs)
        if len(ptrs) != world * n_tasks:
            raise ValueError("dst table must have world * n_tasks entries")
        self.world, self.n_tasks = world, n_tasks
        self.c = (ctypes.c_void_p * max(len(ptrs), 1))(*[p if p else None for p in ptrs])
        self.addr = ctypes.addressof(self.c)

    def nonempty(self) -> np.ndarray:
        return np.array([bool(self.c[i]) for i in range(self.world * self.n_tasks)]).reshape(self.world, self.n_tasks)


def flush_probe(world: int, tasks: np.ndarray, owner, dst: DstTable | None, reduce_to_owner: bool = True,
                flush_index: int = 0) -> Probe:
    t = _tasks_arg(tasks)
    own = None if owner is None else np.ascontiguousarray(owner, dtype=np.int32)
    p = _Probe()
    p.flush_index = flush_index
    _check(lib().dpred_flush_probe(world, t.ctypes.data, len(t), None if own is None else own.ctypes.data,
                                   0 if own is None else len(own), None if dst is None else dst.c,
                                   int(reduce_to_owner), ctypes.byref(p)))
    return _probe_from(p, world)


def flush_workspace_bytes(world: int, n_tasks: int) -> int:
    return int(lib().dpred_flush_workspace_bytes(world, n_tasks))


FLUSH_CHECKED, FLUSH_OVERLAP = 1, 2


def flush_bucket(grads, tasks: np.ndarray, owner, dst: DstTable | None, out_dtype: int | None = None,
                 pre_div: bool = True, reduce_to_owner: bool = True, checked: bool = False, probe: bool = False,
                 flush_index: int = 0, workspace=None, stream=None, overlap: bool = False):
    """grads: CUDA tensor [W, m] (row stride = ld, e.g. a column slice of the
    whole [W, n] gradient); tasks: TASK_DTYPE array; owner: int32 per param or
    None; dst: DstTable or None (in place).  overlap=True promises that this
    flush shares no byte with the work just before it on the stream
    (DPRED_FLUSH_OVERLAP).  Returns a Probe when probe=True."""
    shape, strides = grads.shape, grads.stride()
    if len(shape) != 2 or strides[1] != 1:
        raise ValueError("grads must be a 2-D CUDA tensor with unit column stride")
    world = shape[0]
    in_dt = _dtype_code(grads)
    out_dt = in_dt if out_dtype is None else out_dtype
    ld = strides[0] if world > 1 else shape[1]
    t = _tasks_arg(tasks)
    own = _owner_arg(owner)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                             workspace.numel() * workspace.element_size())
    flags = (FLUSH_CHECKED if checked else 0) | (FLUSH_OVERLAP if overlap else 0)
    fc = _FC if _FC is not None else _fast_call_module()
    if fc is not None:  # the same call through the CPython module (no ctypes conversion)
        r = fc.call(_flush_fn_address(), world, in_dt, grads.data_ptr(), ld, _ptr(t), len(t),
                    0 if own is None else _ptr(own), 0 if own is None else len(own), out_dt,
                    0 if dst is None else dst.addr, 1 if pre_div else 0, 1 if reduce_to_owner else 0, flags,
                    ws_ptr or 0, ws_bytes, _stream(stream), flush_index if probe else None)
        if not probe:
            if r:
                _check(r)
            return None
        if r[0]:
            _check(r[0])
        return Probe(*r[1:])
    p = _Probe() if probe else None
    if p is not None:
        p.flush_index = flush_index
    rc = lib().dpred_flush_bucket(world, in_dt, grads.data_ptr(), ld, _ptr(t), len(t),
                                  None if own is None else _ptr(own), 0 if own is None else len(own),
                                  out_dt, None if dst is None else dst.c, 1 if pre_div else 0,
                                  1 if reduce_to_owner else 0, flags, None if p is None else ctypes.byref(p),
                                  ws_ptr, ws_bytes, _stream(stream))
    if rc:
        _check(rc)
    return _probe_from(p, world) if p is not None else None


_FC = None
_FLUSH_FN = None


def _flush_fn_address() -> int:
    global _FLUSH_FN
    if _FLUSH_FN is None:
        _FLUSH_FN = ctypes.cast(lib().dpred_flush_bucket, ctypes.c_void_p).value
    return _FLUSH_FN


def _fast_call_module():
    """The optional CPython call module (built beside the library when this
    Python has headers), or None; BucketFlush then calls through ctypes."""
    global _FC
    if _FC is None:
        try:
            from . import _fastcall as fc
        except ImportError:
            return None
        _FC = fc
    return _FC


class BucketFlush:
    """One bucket's dpred_flush_bucket call with every argument marshalled
    once: the gradient view, the task table, the owner map, the destination
    table and the options.  A caller that flushes the same bucket every step
    keeps one per bucket; calling it passes only the stream and, when asked,
    a probe, and the library's plan cache serves the validated plan.  The
    arrays it was built from must not be changed afterwards (build a new
    object instead).  The call goes through the small CPython module built
    beside the library where there is one (``fast`` is then True), else
    through ctypes; ``fast=False`` asks for ctypes.  Both reach the same
    dpred_flush_bucket in the same loaded library."""

    def __init__(self, grads, tasks: np.ndarray, owner, dst: DstTable | None, out_dtype: int | None = None,
                 pre_div: bool = True, reduce_to_owner: bool = True, checked: bool = False, overlap: bool = False,
                 workspace=None, fast: bool = True):
        shape, strides = grads.shape, grads.stride()
        if len(shape) != 2 or strides[1] != 1:
            raise ValueError("grads must be a 2-D CUDA tensor with unit column stride")
        self.world = shape[0]
        in_dt = _dtype_code(grads)
        self._tasks = _tasks_arg(tasks).copy()
        self._owner = None if owner is None else np.array(owner, dtype=np.int32, copy=True)
        self._dst = dst
        self._workspace = workspace
        flags = (FLUSH_CHECKED if checked else 0) | (FLUSH_OVERLAP if overlap else 0)
        ld = strides[0] if self.world > 1 else shape[1]
        self._fn = lib().dpred_flush_bucket
        self._head = (self.world, in_dt, grads.data_ptr(), ld, self._tasks.ctypes.data, len(self._tasks),
                      None if self._owner is None else self._owner.ctypes.data,
                      0 if self._owner is None else len(self._owner), in_dt if out_dtype is None else out_dtype,
                      None if dst is None else dst.c, 1 if pre_div else 0, 1 if reduce_to_owner else 0, flags)
        self._ws = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                         workspace.numel() * workspace.element_size())
        self._grads = grads  # keeps the tensor the pointers refer to alive
        fc = _fast_call_module() if fast else None
        if fc is not None:  # the same arguments as integer addresses (0 = NULL)
            head = list(self._head)
            head[9] = 0 if dst is None else ctypes.addressof(dst.c)
            self._cap = fc.prepare(ctypes.cast(self._fn, ctypes.c_void_p).value,
                                   *(0 if a is None else a for a in (*head, *self._ws)))
        else:
            self._cap = None
        self.fast = self._cap is not None

    def __call__(self, stream=None, probe: bool = False, flush_index: int = 0):
        if self._cap is not None:
            if probe:
                r = _FC.flush_probed(self._cap, _stream(stream), flush_index)
                if r[0]:
                    _check(r[0])
                return Probe(*r[1:])
            rc = _FC.flush(self._cap, _stream(stream))
            if rc:
                _check(rc)
            return None
        p = None
        if probe:
            p = _Probe()
            p.flush_index = flush_index
        rc = self._fn(*self._head, None if p is None else ctypes.byref(p), *self._ws, _stream(stream))
        if rc:
            _check(rc)
        return _probe_from(p, self.world) if p is not None else None


def flush_bucket_noalloc(grads, tasks: np.ndarray, owner, dst: DstTable | None, out_dtype: int | None = None,
                         pre_div: bool = True, reduce_to_owner: bool = True, checked: bool = False,
                         probe: bool = False, flush_index: int = 0, stream=None):
    """flush_bucket for callers that cannot allocate device memory (a runtime
    with a fixed device budget, a plug-in inside another framework's
    allocator): no workspace, the library's own 1 MiB scratch holds large task
    tables.  Calls that overlap on the GPU share that scratch, so issue them
    on one stream."""
    if grads.dim() != 2 or grads.stride(1) != 1:
        raise ValueError("grads must be a 2-D CUDA tensor with unit column stride")
    world = grads.shape[0]
    in_dt = _dtype_code(grads)
    out_dt = in_dt if out_dtype is None else out_dtype
    ld = grads.stride(0) if world > 1 else grads.shape[1]
    t = _tasks_arg(tasks)
    own = None if owner is None else np.ascontiguousarray(owner, dtype=np.int32)
    p = _Probe() if probe else None
    if p is not None:
        p.flush_index = flush_index
    _check(lib().dpred_flush_bucket_noalloc(world, in_dt, grads.data_ptr(), ld, t.ctypes.data, len(t),
                                            None if own is None else own.ctypes.data,
                                            0 if own is None else len(own), out_dt,
                                            None if dst is None else dst.c, int(pre_div), int(reduce_to_owner),
                                            int(checked), None if p is None else ctypes.byref(p), _stream(stream)))
    return _probe_from(p, world) if p is not None else None


def flush_bucket_partitioned(grads, tasks: np.ndarray, flat_offset, part_size: int, part_dst, out_dtype: int | None = None,
                             pre_div: bool = True, probe: bool = False, workspace=None, stream=None):
    """Every rank gets its partition's slice of the reduced bucket.  part_dst:
    list of CUDA tensors (each >= part_size elements) or None per rank."""
    if grads.dim() != 2 or grads.stride(1) != 1:
        raise ValueError("grads must be a 2-D CUDA tensor with unit column stride")
    world = grads.shape[0]
    in_dt = _dtype_code(grads)
    out_dt = in_dt if out_dtype is None else out_dtype
    ld = grads.stride(0) if world > 1 else grads.shape[1]
    t = _tasks_arg(tasks)
    fo = np.ascontiguousarray(flat_offset, dtype=np.int64)
    table = (ctypes.c_void_p * world)(*[None if d is None else d.data_ptr() for d in part_dst])
    p = _Probe() if probe else None
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                             workspace.numel() * workspace.element_size())
    _check(lib().dpred_flush_bucket_partitioned(world, in_dt, grads.data_ptr(), ld, t.ctypes.data, len(t),
                                                fo.ctypes.data, len(fo), int(part_size), out_dt, table, int(pre_div),
                                                None if p is None else ctypes.byref(p), ws_ptr, ws_bytes,
                                                _stream(stream)))
    return _probe_from(p, world) if p is not None else None


def bucket_relayout(grads, tasks: np.ndarray, flat_offset, part_size: int, seg: int, out, workspace=None,
                    stream=None) -> np.ndarray:
    """Rank-major relayout of the bucket into out ([W, >= W*seg]); returns the run lengths."""
    if grads.dim() != 2 or grads.stride(1) != 1 or out.dim() != 2 or out.stride(1) != 1:
        raise ValueError("2-D CUDA tensors with unit column stride required")
    world = grads.shape[0]
    t = _tasks_arg(tasks)
    fo = np.ascontiguousarray(flat_offset, dtype=np.int64)
    used = np.zeros(world, np.int64)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                             workspace.numel() * workspace.element_size())
    _check(lib().dpred_bucket_relayout(world, _dtype_code(grads), grads.data_ptr(),
                                       grads.stride(0) if world > 1 else grads.shape[1], t.ctypes.data, len(t),
                                       fo.ctypes.data, len(fo), int(part_size), int(seg), out.data_ptr(),
                                       out.stride(0) if world > 1 else out.shape[1], used.ctypes.data, ws_ptr,
                                       ws_bytes, _stream(stream)))
    return used


def bucket_relayout_workspace_bytes(world: int, n_tasks: int) -> int:
    return int(lib().dpred_bucket_relayout_workspace_bytes(world, n_tasks))


# ----------------------------------------------------- accumulate / RS / AG ---

def accumulate_microbatch(acc, g, first: bool, finalize: bool, scale: float = 1.0, total=None, stream=None):
    """acc: fp32 CUDA tensor [W, n]; g: [W, n] bf16/fp32; total: fp32 [n] when finalize."""
    import torch
    if acc.dtype != torch.float32 or not acc.is_contiguous() or not g.is_contiguous() or acc.shape != g.shape:
        raise ValueError("acc must be contiguous fp32 [W, n] and g contiguous [W, n]")
    if finalize and (total is None or total.dtype != torch.float32 or total.numel() != acc.shape[1]):
        raise ValueError("finalize needs an fp32 total of n elements")
    W, n = acc.shape
    _check(lib().dpred_accumulate_microbatch(W, n, acc.data_ptr(), _dtype_code(g), g.data_ptr(), int(first),
                                             int(finalize), float(scale),
                                             total.data_ptr() if finalize else None, _stream(stream)))
    return total


def accumulator_save(acc, total, stream=None):
    """total = sum over replica rows of acc (the reduced form a checkpoint holds)."""
    import torch
    if acc.dtype != torch.float32 or total.dtype != torch.float32 or not acc.is_contiguous() \
            or total.numel() != acc.shape[1]:
        raise ValueError("acc: contiguous fp32 [W, n]; total: fp32 [n]")
    W, n = acc.shape
    _check(lib().dpred_accumulator_save(W, n, acc.data_ptr(), total.data_ptr(), _stream(stream)))
    return total


def accumulator_restore(acc, total, stream=None):
    """acc[0] = total, acc[1:] = 0 (the unreduced form of a restored total)."""
    import torch
    if acc.dtype != torch.float32 or total.dtype != torch.float32 or not acc.is_contiguous() \
            or total.numel() != acc.shape[1]:
        raise ValueError("acc: contiguous fp32 [W, n]; total: fp32 [n]")
    W, n = acc.shape
    _check(lib().dpred_accumulator_restore(W, n, acc.data_ptr(), total.data_ptr(), _stream(stream)))
    return acc


def reduce_scatter(inp, out, pre_div: bool = False, stream=None):
    """inp: CUDA tensor [N, M]; out: [N, M/N] (bf16 or fp32)."""
    if not inp.is_contiguous() or not out.is_contiguous():
        raise ValueError("contiguous tensors required")
    N, M = inp.shape
    _check(lib().dpred_reduce_scatter(N, M, _dtype_code(inp), inp.data_ptr(), _dtype_code(out), out.data_ptr(),
                                      int(pre_div), _stream(stream)))
    return out


def allgather(inp, out, order: int = 0, stream=None):
    """inp: CUDA tensor [N, S]; out: [N, N*S] of the same dtype; order 0 canonical, 1 ring."""
    if not inp.is_contiguous() or not out.is_contiguous() or inp.dtype != out.dtype:
        raise ValueError("contiguous tensors of one dtype required")
    N, S = inp.shape
    if tuple(out.shape) != (N, N * S):
        raise ValueError("out must be [N, N*S]")
    _check(lib().dpred_allgather(N, S, _dtype_code(inp), inp.data_ptr(), out.data_ptr(), int(order),
                                 _stream(stream)))
    return out


PATH_AUTO, PATH_LDG, PATH_TMA = 0, 1, 2


def set_flush_path(path: int) -> int:
    """Kernel family of later flushes: PATH_AUTO, PATH_LDG or PATH_TMA.  Returns the previous one."""
    rc = lib().dpred_set_flush_path(int(path))
    if rc < 0:
        _check(rc)
    return rc


AG_AUTO, AG_REGISTER, AG_TMA1, AG_TMA4, AG_STAGED, AG_SKEW, AG_SKEW8K = 0, 1, 2, 3, 4, 5, 6


def set_allgather_form(form: int) -> int:
    """Kernel form of later AllGathers (AG_*, see dpred_set_allgather_form).  Returns the previous one."""
    rc = lib().dpred_set_allgather_form(int(form))
    if rc < 0:
        _check(rc)
    return rc


def fill_pattern(t, pattern: int = 0, method: int = 0, ctas_per_sm: int = 0, stream=None):
    """Write-only fill of a CUDA tensor's bytes (dpred_fill_pattern: the HBM write ceiling)."""
    _check(lib().dpred_fill_pattern(t.data_ptr(), t.numel() * t.element_size(), int(pattern) & 0xFFFFFFFF,
                                    int(method), int(ctas_per_sm), _stream(stream)))
    return t


def stream_mixed(src, dst, read_bytes: int | None = None, write_bytes: int | None = None, stream=None):
    """Read src and write dst concurrently with no dependency (dpred_stream_mixed:
    the HBM ceiling for that mix of reads and writes)."""
    rb = src.numel() * src.element_size() if read_bytes is None else int(read_bytes)
    wb = dst.numel() * dst.element_size() if write_bytes is None else int(write_bytes)
    _check(lib().dpred_stream_mixed(src.data_ptr(), rb, dst.data_ptr(), wb, _stream(stream)))


def selftest_wait_timeout(budget_cycles: int = 2_000_000, stream=None) -> None:
    """Launch a kernel whose bounded wait must give up (see dpred_selftest_wait_timeout)."""
    _check(lib().dpred_selftest_wait_timeout(int(budget_cycles), _stream(stream)))


SCHED_RING, SCHED_BIDIR_RING, SCHED_RECURSIVE_DOUBLING = 0, 1, 2


def allgather_schedule_steps(schedule: int, n_nodes: int) -> int:
    rc = lib().dpred_allgather_schedule_steps(schedule, n_nodes)
    if rc < 0:
        _check(rc)
    return rc


def allgather_schedule_init(schedule: int, inp, bufs, stream=None):
    """inp: [N, S] shards; bufs: [N, N*S] node buffers (same dtype)."""
    N, S = inp.shape
    if tuple(bufs.shape) != (N, N * S) or bufs.dtype != inp.dtype or not bufs.is_contiguous() \
            or not inp.is_contiguous():
        raise ValueError("bufs must be contiguous [N, N*S] of the shards' dtype")
    _check(lib().dpred_allgather_schedule_init(schedule, N, S, _dtype_code(inp), inp.data_ptr(), bufs.data_ptr(),
                                               _stream(stream)))


def allgather_schedule_step(schedule: int, bufs, step: int, stream=None):
    N = bufs.shape[0]
    _check(lib().dpred_allgather_schedule_step(schedule, N, bufs.shape[1] // N, _dtype_code(bufs), bufs.data_ptr(),
                                               int(step), _stream(stream)))


def checked_build() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(lib().dpred_checked_build())


def selftest_prediv(world: int) -> tuple[int, int]:
    """(mismatches, lowest mismatching fp32 bit pattern or 0xFFFFFFFF) of the
    flush's pre-division by `world` against IEEE division, over every fp32
    input (dpred_selftest_prediv)."""
    n, f = ctypes.c_uint64(), ctypes.c_uint32()
    _check(lib().dpred_selftest_prediv(int(world), ctypes.byref(n), ctypes.byref(f)))
    return int(n.value), int(f.value)


def selftest_bounds(stream=None) -> None:
    _check(lib().dpred_selftest_bounds(_stream(stream)))


def device_status(clear: bool = False) -> int:
    code = ctypes.c_int32()
    _check(lib().dpred_device_status(ctypes.byref(code), int(clear)))
    return code.value


def host_mapped_pointer(t) -> int:
    """Device address of a pinned host tensor's first element (the address a
    kernel uses to read or write it over the host link)."""
    out = ctypes.c_void_p()
    _check(lib().dpred_host_mapped_pointer(t.data_ptr(), ctypes.byref(out)))
    return int(out.value or 0)


# ------------------------------------------------------- gradient buffers ---

class GradBuffers:
    """Real gradient buffers on the ranks that hold a parameter, nothing on the
    others (the DeepSpeed issue: a real buffer only on the rank whose optimizer
    partition holds the parameter, ``torch.empty([0])`` everywhere else; a
    straddling parameter is held by every rank of its partition range).

    One flat CUDA tensor per rank; each held parameter gets a slot whose start
    keeps the parameter's offset in the gradient row modulo 16 bytes, so the
    flush can use 16-byte vectors for it."""

    def __init__(self, world: int, omap: OwnerMap, numel, row_offset, dtype, device="cuda", fill=None):
        import torch
        self.world = world
        esize = 2 if dtype == torch.bfloat16 else 4
        per = 16 // esize
        numel = np.asarray(numel, dtype=np.int64)
        row_offset = np.asarray(row_offset, dtype=np.int64)
        self.slot = [dict() for _ in range(world)]
        sizes = [0] * world
        for p in range(len(numel)):
            lo, hi = int(omap.holder_lo[p]), int(omap.holder_hi[p])
            if lo < 0 or numel[p] == 0:
                continue
            for r in range(lo, hi + 1):
                start = sizes[r]
                start += (int(row_offset[p]) - start) % per  # co-align with the gradient row
                self.slot[r][p] = start
                sizes[r] = start + int(numel[p])
        self.buf = []
        for r in range(world):
            t = torch.empty(max(sizes[r], 1), dtype=dtype, device=device)
            if fill is not None:
                t.fill_(fill)
            self.buf.append(t)
        self.numel = numel
        self.esize = esize

    def view(self, rank: int, param: int):
        """Rank ``rank``'s buffer for ``param`` (None when it holds none)."""
        s = self.slot[rank].get(param)
        if s is None:
            return None
        return self.buf[rank][s:s + int(self.numel[param])]

    def dst_table(self, tasks: np.ndarray) -> DstTable:
        n = len(tasks)
        ptrs = [0] * (self.world * n)
        for t, task in enumerate(tasks):
            p = int(task["param_id"])
            for r in range(self.world):
                s = self.slot[r].get(p)
                if s is not None:
                    ptrs[r * n + t] = self.buf[r].data_ptr() + s * self.esize
        return DstTable(self.world, n, ptrs)


# ------------------------------------------------------- ZeRO-1 executor ---

class Zero1Executor:
    """The ZeRO-1 bucket-flush executor (dpred_executor_*): the owner map, the
    installed gradient buffers and every bucket's prebuilt launch plan; a step
    is one native call that flushes every bucket in order (the DeepSpeed
    issue's Z1CustomOpExecutor::flushReduceBucket, with the collective replaced
    by the single-GPU kernel).

    buckets: list of (start, tasks) -- the bucket's element offset in the
    arrival-order gradient row and its TASK_DTYPE task table.  The native
    executor is bound to the gradient tensor of the first flush (and rebuilt
    if a different tensor is passed)."""

    def __init__(self, world: int, numel, row_offset, buckets, dtype, reduce_to_owner: bool = True,
                 pre_div: bool = True, groups=None, probe_log: ProbeLog | None = None, fill=None):
        import torch
        self.world = world
        self.dtype = dtype
        self.dt_code = BF16 if dtype == torch.bfloat16 else F32
        self.reduce_to_owner, self.pre_div = reduce_to_owner, pre_div
        groups = [(None, numel)] if groups is None else groups
        self.omap = build_owner_map(world, groups, reduce_to_owner)
        self.grad = GradBuffers(world, self.omap, numel, row_offset, dtype, fill=fill)
        self.buckets = [(int(s), np.ascontiguousarray(t, dtype=TASK_DTYPE)) for s, t in buckets]
        self.tables = [self.grad.dst_table(t) for _, t in self.buckets]
        self.sizes = [int((t["offset"] + t["numel"]).max()) if len(t) else 0 for _, t in self.buckets]
        self.probe_log = probe_log
        ws = max((flush_workspace_bytes(world, len(t)) for _, t in self.buckets), default=0)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device="cuda") if ws else None
        self.overlap = True
        self._native = None
        self._bound = None

    def _bind(self, grads):
        if grads.dim() != 2 or grads.stride(1) != 1 or grads.shape[0] != self.world:
            raise ValueError("grads must be a [W, n] CUDA tensor with unit column stride")
        ld = grads.stride(0) if self.world > 1 else grads.shape[1]
        key = (grads.data_ptr(), ld, grads.dtype)
        if self._bound == key:
            return
        self.close()
        nb = len(self.buckets)
        tasks = np.ascontiguousarray(np.concatenate([t for _, t in self.buckets]) if nb else np.zeros(0, TASK_DTYPE))
        starts = np.array([s for s, _ in self.buckets], np.int64)
        counts = np.array([len(t) for _, t in self.buckets], np.int32)
        handle = ctypes.c_void_p()
        ws_ptr, ws_bytes = (None, 0) if self.workspace is None else (self.workspace.data_ptr(), self.workspace.numel())
        self._create(grads, ld, nb, starts, counts, tasks, ws_ptr, ws_bytes, handle)
        self._native = handle
        self._bound = key
        lib().dpred_executor_set_overlap(self._native, int(self.overlap))

    def _create(self, grads, ld, nb, starts, counts, tasks, ws_ptr, ws_bytes, handle):
        total = sum(self.world * len(t) for _, t in self.buckets)
        dst = (ctypes.c_void_p * max(total, 1))()
        pos = 0
        for tab in self.tables:
            n = tab.world * tab.n_tasks
            for i in range(n):
                dst[pos + i] = tab.c[i]
            pos += n
        _check(lib().dpred_executor_create(self.world, _dtype_code(grads), self.dt_code, int(self.pre_div),
                                           int(self.reduce_to_owner), self.omap.owner.ctypes.data, len(self.omap.owner),
                                           grads.data_ptr(), ld, nb, starts.ctypes.data, counts.ctypes.data,
                                           tasks.ctypes.data, dst, ws_ptr, ws_bytes, ctypes.byref(handle)))

    def _regions(self):
        """The device buffers the step writes into, one per rank."""
        return self.grad.buf

    def set_overlap(self, on: bool) -> bool:
        """Let consecutive bucket flushes of a step overlap on the GPU (the
        default; used only when the buckets share no byte).  Returns the
        previous setting."""
        prev, self.overlap = self.overlap, bool(on)
        if self._native is not None:
            lib().dpred_executor_set_overlap(self._native, int(self.overlap))
        return prev

    def close(self):
        if self._native is not None and _lib is not None:
            lib().dpred_executor_destroy(self._native)
        self._native = None
        self._bound = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _probes(self, want: bool):
        return (_Probe * max(len(self.buckets), 1))() if want else None

    def _finish(self, probes, probe: bool):
        if probes is None:
            return None
        out = [_probe_from(probes[b], self.world) for b in range(len(self.buckets))]
        if self.probe_log is not None:
            for p in out:
                self.probe_log.record(p, self.dt_code, self.pre_div)
        return out if probe else None

    def flush_all(self, grads, stream=None, probe: bool = False):
        """Flush every bucket of grads ([W, n], arrival-order rows) on a stream.
        Returns the probes when probe=True."""
        self._bind(grads)
        probes = self._probes(probe or self.probe_log is not None)
        _check(lib().dpred_executor_flush_all(self._native, probes, _stream(stream)))
        return self._finish(probes, probe)

    def flush_bucket(self, grads, bucket: int, stream=None):
        self._bind(grads)
        _check(lib().dpred_executor_flush(self._native, int(bucket), None, _stream(stream)))

    def flush_all_from_host(self, host_grads, host_bufs, grads, stream=None, probe: bool = False):
        """One step with host buffers: host_grads (pinned [W, n]) is copied into
        grads bucket by bucket, every bucket is flushed, and each rank's
        gradient buffer is copied back into host_bufs[r] (pinned, same size),
        pipelined over buckets on the executor's copy streams."""
        self._bind(grads)
        W = self.world
        if len(host_bufs) != W:
            raise ValueError("one host buffer per rank")
        dev = (ctypes.c_void_p * W)(*[b.data_ptr() for b in self._regions()])
        host = (ctypes.c_void_p * W)(*[h.data_ptr() for h in host_bufs])
        nbytes = np.array([b.numel() * b.element_size() for b in self._regions()], np.int64)
        for h, n in zip(host_bufs, nbytes):
            if h.numel() * h.element_size() < n:
                raise ValueError("host buffer smaller than its device buffer")
        probes = self._probes(probe or self.probe_log is not None)
        hld = host_grads.stride(0) if W > 1 else host_grads.shape[1]
        _check(lib().dpred_executor_flush_all_from_host(self._native, host_grads.data_ptr(), hld, W, dev, host,
                                                        nbytes.ctypes.data, probes, _stream(stream)))
        return self._finish(probes, probe)

    def flush_all_mapped(self, host_grads, host_bufs, grads, stream=None, probe: bool = False):
        """The host-buffer step without staging: the flush kernels read
        host_grads (pinned [W, n]) and write each rank's reduced gradients into
        host_bufs[r] (pinned, laid out like that rank's device buffer) over the
        host link.  grads and the device buffers are not touched."""
        self._bind(grads)
        W = self.world
        if len(host_bufs) != W:
            raise ValueError("one host buffer per rank")
        for h, b in zip(host_bufs, self._regions()):
            if h.numel() * h.element_size() < b.numel() * b.element_size():
                raise ValueError("host buffer smaller than its device buffer")
        dev = (ctypes.c_void_p * W)(*[b.data_ptr() for b in self._regions()])
        host = (ctypes.c_void_p * W)(*[h.data_ptr() for h in host_bufs])
        nbytes = np.array([b.numel() * b.element_size() for b in self._regions()], np.int64)
        probes = self._probes(probe or self.probe_log is not None)
        hld = host_grads.stride(0) if W > 1 else host_grads.shape[1]
        _check(lib().dpred_executor_flush_all_mapped(self._native, host_grads.data_ptr(), hld, W, dev, host,
                                                     nbytes.ctypes.data, probes, _stream(stream)))
        return self._finish(probes, probe)


class InPlaceExecutor(Zero1Executor):
    """The executor in place (dpred_executor_create with no destination
    table): every flush writes its delivered results back into the gradient
    rows themselves, row owner(t) for an owned parameter and every row for an
    AllReduce one, as a bucket's collective does on the bucket's own memory.
    The probes count what each row received.  A step is one native call with
    launch overlap between buckets (in-place writes stay inside their own
    bucket's columns); the host-buffer steps need destination buffers and are
    not available."""

    def __init__(self, world: int, numel, buckets, dtype, reduce_to_owner: bool = True, pre_div: bool = True,
                 groups=None, probe_log: ProbeLog | None = None):
        import torch
        self.world = world
        self.dtype = dtype
        self.dt_code = BF16 if dtype == torch.bfloat16 else F32
        self.reduce_to_owner, self.pre_div = reduce_to_owner, pre_div
        groups = [(None, numel)] if groups is None else groups
        self.omap = build_owner_map(world, groups, reduce_to_owner)
        self.grad = None
        self.buckets = [(int(s), np.ascontiguousarray(t, dtype=TASK_DTYPE)) for s, t in buckets]
        self.sizes = [int((t["offset"] + t["numel"]).max()) if len(t) else 0 for _, t in self.buckets]
        self.probe_log = probe_log
        ws = max((flush_workspace_bytes(world, len(t)) for _, t in self.buckets), default=0)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device="cuda") if ws else None
        self.overlap = True
        self._native = None
        self._bound = None

    def _create(self, grads, ld, nb, starts, counts, tasks, ws_ptr, ws_bytes, handle):
        if _dtype_code(grads) != self.dt_code:
            raise TypeError("an in-place executor keeps the gradient dtype")
        _check(lib().dpred_executor_create(self.world, _dtype_code(grads), self.dt_code, int(self.pre_div),
                                           int(self.reduce_to_owner), self.omap.owner.ctypes.data, len(self.omap.owner),
                                           grads.data_ptr(), ld, nb, starts.ctypes.data, counts.ctypes.data,
                                           tasks.ctypes.data, None, ws_ptr, ws_bytes, ctypes.byref(handle)))

    def _regions(self):
        raise DpredError(-1, "host-buffer steps need destination buffers (in-place executor)")


class PartitionedExecutor(Zero1Executor):
    """The executor over partitioned flushes (dpred_executor_create_partitioned):
    every rank receives exactly its own partition of the reduced gradients,
    the ReduceScatter form of the DeepSpeed issue's "better end state" and the
    ZeRO-2 follow-up (real buffers with offsets).  The flat (model-order)
    space of all parameters is cut into W partitions of P = ceil(T / W)
    elements; ``parts[r]`` is rank r's partition buffer (P elements).  A step
    is one native call, with the same launch overlap and host-buffer steps as
    Zero1Executor (the host buffers then mirror ``parts``)."""

    def __init__(self, world: int, numel, row_offset, buckets, dtype, pre_div: bool = True,
                 probe_log: ProbeLog | None = None, parts=None):
        import torch
        self.world = world
        self.dtype = dtype
        self.dt_code = BF16 if dtype == torch.bfloat16 else F32
        self.reduce_to_owner, self.pre_div = True, pre_div
        numel = np.asarray(numel, np.int64)
        self.flat_offset = np.concatenate([[0], np.cumsum(numel)[:-1]]).astype(np.int64)
        total = int(numel.sum())
        self.part_size = max(-(-total // world), 1)
        self.parts = parts if parts is not None else \
            [torch.empty(self.part_size, dtype=dtype, device="cuda") for _ in range(world)]
        if len(self.parts) != world or any(p.numel() < self.part_size for p in self.parts):
            raise ValueError(f"one partition buffer of {self.part_size} elements per rank")
        self.buckets = [(int(s), np.ascontiguousarray(t, dtype=TASK_DTYPE)) for s, t in buckets]
        self.sizes = [int((t["offset"] + t["numel"]).max()) if len(t) else 0 for _, t in self.buckets]
        self.probe_log = probe_log
        # a task is cut into at most (pieces it spans) destinations: n_tasks + world - 1 per bucket
        ws = max((flush_workspace_bytes(world, len(t) + world) for _, t in self.buckets), default=0)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device="cuda") if ws else None
        self.overlap = True
        self._native = None
        self._bound = None

    def _create(self, grads, ld, nb, starts, counts, tasks, ws_ptr, ws_bytes, handle):
        W = self.world
        parts = (ctypes.c_void_p * W)(*[p.data_ptr() for p in self.parts])
        _check(lib().dpred_executor_create_partitioned(W, _dtype_code(grads), self.dt_code, int(self.pre_div),
                                                       grads.data_ptr(), ld, nb, starts.ctypes.data, counts.ctypes.data,
                                                       tasks.ctypes.data, self.flat_offset.ctypes.data,
                                                       len(self.flat_offset), self.part_size, parts, ws_ptr, ws_bytes,
                                                       ctypes.byref(handle)))

    def _regions(self):
        return self.parts
