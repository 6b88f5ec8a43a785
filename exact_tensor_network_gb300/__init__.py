"""GB300 executor for exact tensor-network contraction along a fixed tree.

Thin ctypes binding of the C ABI in ``include/tn.h`` (``libtn_gb300.so``,
built in-tree by ``exact_tensor_network_gb300.build``).  The functions below
carry the C names and only marshal arguments; every step of the contraction
runs in the library's CUDA kernels.  PyTorch is used for device memory and
streams only.  There is no fallback: if the library is not built, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtn_gb300.so")

# status codes (tn_status)
TN_OK, TN_EINVAL, TN_ENOMEM, TN_EOVERFLOW, TN_ECUDA, TN_EDEVICE, TN_ETIMEOUT, TN_ENOTIMPL = range(8)
# precisions
TN_PREC_TF32X3, TN_PREC_BF16, TN_PREC_FP32, TN_PREC_BF16X3 = 0, 1, 2, 3
PRECISIONS = {"tf32x3": TN_PREC_TF32X3, "bf16": TN_PREC_BF16, "fp32": TN_PREC_FP32,
              "bf16x3": TN_PREC_BF16X3}
# node classes
TN_NODE_SIMT, TN_NODE_DENSE, TN_NODE_STREAM, TN_NODE_TINY, TN_NODE_FUSED = 0, 1, 2, 3, 4
NODE_CLASS_NAMES = {0: "simt", 1: "dense", 2: "stream", 3: "tiny", 4: "fused"}
# policies
TN_POLICY_AUTO, TN_POLICY_SIMT, TN_POLICY_NO_TINY = 0, 1, 2
# test setting outside the C ABI: every node the tensor-core kernel can take
# goes there (deep chains of such nodes are not held to the complex64
# tolerance)
TN_POLICY_DENSE = 3


class TNError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


class tn_network(ctypes.Structure):
    _fields_ = [("n_tensors", ctypes.c_int32),
                ("ranks", ctypes.POINTER(ctypes.c_int32)),
                ("modes", ctypes.POINTER(ctypes.POINTER(ctypes.c_int32))),
                ("n_modes", ctypes.c_int32),
                ("extents", ctypes.POINTER(ctypes.c_int64)),
                ("n_open", ctypes.c_int32),
                ("open_modes", ctypes.POINTER(ctypes.c_int32)),
                ("precision", ctypes.c_int32)]


class tn_tree(ctypes.Structure):
    _fields_ = [("n_steps", ctypes.c_int32), ("pairs", ctypes.POINTER(ctypes.c_int32))]


class tn_launch_record(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("step", ctypes.c_int32), ("ms", ctypes.c_float),
                ("flops", ctypes.c_uint64), ("bytes", ctypes.c_uint64)]


KERNEL_NAMES = {0: "permute", 1: "simt", 2: "dense_tf32x3", 3: "dense_bf16", 4: "stream", 5: "tiny",
                6: "reduce", 7: "dense_tf32x3_3p", 8: "dense_bf16x3", 9: "fused"}


class tn_slices(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("modes", ctypes.POINTER(ctypes.c_int32))]


_lib = None
_P = ctypes.c_void_p
_U64P = ctypes.POINTER(ctypes.c_uint64)
_I32P = ctypes.POINTER(ctypes.c_int32)

# exported symbol -> (restype, argtypes)
SIGNATURES = {
    "tn_plan": (ctypes.c_int, [ctypes.POINTER(tn_network), ctypes.POINTER(tn_tree),
                               ctypes.POINTER(tn_slices), ctypes.POINTER(_P)]),
    "tn_plan_destroy": (None, [_P]),
    "tn_plan_flops": (ctypes.c_int, [_P, _U64P]),
    "tn_plan_peak": (ctypes.c_int, [_P, _U64P]),
    "tn_plan_num_slices": (ctypes.c_int, [_P, _U64P]),
    "tn_plan_num_steps": (ctypes.c_int, [_P, _I32P]),
    "tn_plan_mode_order": (ctypes.c_int, [_P, ctypes.c_int32, _I32P, ctypes.c_int32, _I32P]),
    "tn_plan_node_mnk": (ctypes.c_int, [_P, ctypes.c_int32, _U64P]),
    "tn_plan_node_class": (ctypes.c_int, [_P, ctypes.c_int32, _I32P]),
    "tn_plan_set_policy": (ctypes.c_int, [_P, ctypes.c_int32]),
    "tn_plan_workspace_bytes": (ctypes.c_int, [_P, _U64P]),
    "tn_plan_set_workspace": (ctypes.c_int, [_P, _P, ctypes.c_uint64]),
    "tn_execute": (ctypes.c_int, [_P, ctypes.POINTER(_P), _P, _P]),
    "tn_execute_static": (ctypes.c_int, [_P, ctypes.POINTER(_P), _P, _P]),
    "tn_plan_set_replay": (ctypes.c_int, [_P, ctypes.c_int32]),
    "tn_plan_set_three_products": (ctypes.c_int, [_P, ctypes.c_int32]),
    "tn_plan_set_hoisting": (ctypes.c_int, [_P, ctypes.c_int32]),
    "tn_plan_set_fusion": (ctypes.c_int, [_P, ctypes.c_int32]),
    "tn_plan_set_cta_pairs": (ctypes.c_int, [_P, ctypes.c_int32]),
    "tn_plan_set_promotion_chunk": (ctypes.c_int, [_P, ctypes.c_int32]),
    "tn_execute_slices": (ctypes.c_int, [_P, ctypes.POINTER(_P), _P, _P, ctypes.c_uint64,
                                         ctypes.c_uint64]),
    "tn_execute_host": (ctypes.c_int, [_P, ctypes.POINTER(_P), _P, ctypes.POINTER(_P), _P, _P]),
    "tn_plan_check": (ctypes.c_int, [_P]),
    "tn_execute_prefix": (ctypes.c_int, [_P, ctypes.POINTER(_P), _P, ctypes.c_int32, _P]),
    "tn_plan_tensor_gather": (ctypes.c_int, [_P, ctypes.c_int32, _P, ctypes.c_uint64, _P, _P]),
    "tn_plan_launches": (ctypes.c_int, [_P, _U64P]),
    "tn_plan_set_profiling": (ctypes.c_int, [_P, ctypes.c_int32]),
    "tn_plan_profile_read": (ctypes.c_int, [_P, ctypes.POINTER(tn_launch_record), ctypes.c_int32,
                                            _I32P]),
    "tn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tn_last_error": (ctypes.c_char_p, [_P]),
}


def lib() -> ctypes.CDLL:
    """Load libtn_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with exact_tensor_network_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(st: int, plan=None) -> None:
    if st != TN_OK:
        L = lib()
        msg = L.tn_last_error(plan)
        text = (msg.decode() if msg else "") or L.tn_status_string(st).decode()
        raise TNError(st, text)


# ---- functions with the C names -------------------------------------------

def tn_plan(tensors: Sequence[Sequence[int]], extents: Sequence[int],
            open_modes: Sequence[int], pairs: Sequence[Tuple[int, int]],
            slices: Sequence[int] = (), precision: int = TN_PREC_TF32X3) -> int:
    """Plan a contraction; returns the plan handle (an integer)."""
    L = lib()
    n = len(tensors)
    ranks = (ctypes.c_int32 * max(n, 1))(*[len(t) for t in tensors])
    rows = [(ctypes.c_int32 * max(len(t), 1))(*t) for t in tensors]
    mp = (ctypes.POINTER(ctypes.c_int32) * max(n, 1))(
        *[ctypes.cast(r, ctypes.POINTER(ctypes.c_int32)) for r in rows])
    ext = (ctypes.c_int64 * max(len(extents), 1))(*[int(e) for e in extents])
    op = (ctypes.c_int32 * max(len(open_modes), 1))(*[int(x) for x in open_modes])
    net = tn_network(n, ranks, mp, len(extents), ext, len(open_modes), op, int(precision))
    flat = [int(i) for p in pairs for i in p]
    pr = (ctypes.c_int32 * max(len(flat), 1))(*flat)
    tree = tn_tree(len(pairs), pr)
    sm = (ctypes.c_int32 * max(len(slices), 1))(*[int(x) for x in slices])
    sl = tn_slices(len(slices), sm)
    out = _P()
    _check(L.tn_plan(ctypes.byref(net), ctypes.byref(tree), ctypes.byref(sl), ctypes.byref(out)))
    return out.value


def tn_plan_destroy(plan: int) -> None:
    lib().tn_plan_destroy(plan)


def _u64(fn, plan) -> int:
    v = ctypes.c_uint64()
    _check(fn(plan, ctypes.byref(v)), plan)
    return v.value


def tn_plan_flops(plan: int) -> int:
    return _u64(lib().tn_plan_flops, plan)


def tn_plan_peak(plan: int) -> int:
    return _u64(lib().tn_plan_peak, plan)


def tn_plan_num_slices(plan: int) -> int:
    return _u64(lib().tn_plan_num_slices, plan)


def tn_plan_num_steps(plan: int) -> int:
    v = ctypes.c_int32()
    _check(lib().tn_plan_num_steps(plan, ctypes.byref(v)), plan)
    return v.value


def tn_plan_mode_order(plan: int, tensor_id: int):
    ln = ctypes.c_int32()
    _check(lib().tn_plan_mode_order(plan, tensor_id, None, 0, ctypes.byref(ln)), plan)
    buf = (ctypes.c_int32 * max(ln.value, 1))()
    _check(lib().tn_plan_mode_order(plan, tensor_id, buf, ln.value, ctypes.byref(ln)), plan)
    return [buf[i] for i in range(ln.value)]


def tn_plan_node_mnk(plan: int, step: int) -> Tuple[int, int, int]:
    v = (ctypes.c_uint64 * 3)()
    _check(lib().tn_plan_node_mnk(plan, step, v), plan)
    return (v[0], v[1], v[2])


def tn_plan_node_class(plan: int, step: int) -> int:
    v = ctypes.c_int32()
    _check(lib().tn_plan_node_class(plan, step, ctypes.byref(v)), plan)
    return v.value


def tn_plan_set_policy(plan: int, policy: int) -> None:
    _check(lib().tn_plan_set_policy(plan, policy), plan)


def tn_plan_workspace_bytes(plan: int) -> int:
    return _u64(lib().tn_plan_workspace_bytes, plan)


def tn_plan_set_workspace(plan: int, dev_ptr: int, nbytes: int) -> None:
    _check(lib().tn_plan_set_workspace(plan, dev_ptr, nbytes), plan)


def tn_execute(plan: int, leaf_ptrs: Sequence[int], out_ptr: int, stream: int = 0) -> None:
    arr = (_P * max(len(leaf_ptrs), 1))(*leaf_ptrs)
    _check(lib().tn_execute(plan, arr, out_ptr, stream), plan)


def tn_execute_static(plan: int, leaf_ptrs: Sequence[int], out_ptr: int, stream: int = 0) -> None:
    """tn_execute on the library's fixed device scratch array, for callers
    that cannot allocate device memory (no workspace needed; see tn.h)."""
    arr = (_P * max(len(leaf_ptrs), 1))(*leaf_ptrs)
    _check(lib().tn_execute_static(plan, arr, out_ptr, stream), plan)


def tn_execute_slices(plan: int, leaf_ptrs: Sequence[int], out_ptr: int, stream: int,
                      first: int, step: int) -> None:
    arr = (_P * max(len(leaf_ptrs), 1))(*leaf_ptrs)
    _check(lib().tn_execute_slices(plan, arr, out_ptr, stream, first, step), plan)


def tn_execute_host(plan: int, host_leaf_ptrs: Sequence[int], host_out: int,
                    dev_leaf_ptrs: Sequence[int], dev_out: int, stream: int) -> None:
    h = (_P * max(len(host_leaf_ptrs), 1))(*host_leaf_ptrs)
    d = (_P * max(len(dev_leaf_ptrs), 1))(*dev_leaf_ptrs)
    _check(lib().tn_execute_host(plan, h, host_out, d, dev_out, stream), plan)


def tn_execute_prefix(plan: int, leaf_ptrs: Sequence[int], out_ptr: int, step: int,
                      stream: int = 0) -> None:
    arr = (_P * max(len(leaf_ptrs), 1))(*leaf_ptrs)
    _check(lib().tn_execute_prefix(plan, arr, out_ptr, step, stream), plan)


def tn_plan_tensor_gather(plan: int, tensor_id: int, idx_ptr: int, count: int, dst_ptr: int,
                          stream: int = 0) -> None:
    _check(lib().tn_plan_tensor_gather(plan, tensor_id, idx_ptr, count, dst_ptr, stream), plan)


def shard_slices(n_slices: int, rank: int, world: int) -> Tuple[int, int, int]:
    """Slices of rank `rank` among `world` processes: (first, step, count)
    with slices first, first + step, ... below n_slices (round robin).  The
    ranks' outputs add up to the full result."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    count = 0 if rank >= n_slices else (n_slices - 1 - rank) // world + 1
    return rank, world, count


def tn_plan_set_replay(plan: int, enable: bool) -> None:
    _check(lib().tn_plan_set_replay(plan, 1 if enable else 0), plan)


def tn_plan_set_three_products(plan: int, enable: bool) -> None:
    _check(lib().tn_plan_set_three_products(plan, 1 if enable else 0), plan)


def tn_plan_set_hoisting(plan: int, enable: bool) -> None:
    _check(lib().tn_plan_set_hoisting(plan, 1 if enable else 0), plan)


def tn_plan_set_promotion_chunk(plan: int, chunk_k: int) -> None:
    _check(lib().tn_plan_set_promotion_chunk(plan, int(chunk_k)), plan)


def tn_plan_set_cta_pairs(plan: int, enable: bool) -> None:
    _check(lib().tn_plan_set_cta_pairs(plan, 1 if enable else 0), plan)


def tn_plan_set_fusion(plan: int, enable: bool) -> None:
    _check(lib().tn_plan_set_fusion(plan, 1 if enable else 0), plan)


def tn_plan_check(plan: int) -> None:
    _check(lib().tn_plan_check(plan), plan)


def tn_plan_launches(plan: int) -> int:
    return _u64(lib().tn_plan_launches, plan)


def tn_plan_set_profiling(plan: int, enable: bool) -> None:
    _check(lib().tn_plan_set_profiling(plan, 1 if enable else 0), plan)


def tn_plan_profile_read(plan: int):
    """Launch records of the last profiled execute: list of dicts."""
    ln = ctypes.c_int32()
    _check(lib().tn_plan_profile_read(plan, None, 0, ctypes.byref(ln)), plan)
    buf = (tn_launch_record * max(ln.value, 1))()
    _check(lib().tn_plan_profile_read(plan, buf, ln.value, ctypes.byref(ln)), plan)
    return [{"kernel": KERNEL_NAMES.get(r.kernel, str(r.kernel)), "step": r.step, "ms": r.ms,
             "flops": r.flops, "bytes": r.bytes} for r in buf[:ln.value]]


def tn_status_string(status: int) -> str:
    return lib().tn_status_string(status).decode()


def tn_last_error(plan: Optional[int] = None) -> str:
    return lib().tn_last_error(plan).decode()


# ---- convenience wrapper over torch tensors --------------------------------

def _prod(xs) -> int:
    r = 1
    for x in xs:
        r *= x
    return r


def _check_buffers(plan: "Plan", leaves, out, on_device: bool, what: str) -> None:
    """dtype, contiguity, device side and entry counts of the leaves and the
    result against the plan (a short buffer would be read or written past
    its end by the kernels)."""
    import torch
    if len(leaves) != plan.n_tensors:
        raise ValueError(f"{what}: {len(leaves)} leaves given, the network has {plan.n_tensors}")
    where = "CUDA" if on_device else "CPU"
    for t in list(leaves) + [out]:
        if t.dtype != torch.complex64 or not t.is_contiguous() or t.is_cuda != on_device:
            raise ValueError(f"{what}: leaves and result must be contiguous complex64 {where} tensors")
    for i, (t, size) in enumerate(zip(leaves, plan.leaf_sizes)):
        if t.numel() != size:
            raise ValueError(f"{what}: leaf {i} has {t.numel()} entries, its modes give {size}")
    if out.numel() != plan.out_size:
        raise ValueError(f"{what}: result has {out.numel()} entries, the open modes give "
                         f"{plan.out_size}")


class Plan:
    """Owns a plan handle and (optionally) a torch workspace tensor."""

    def __init__(self, tensors, extents, open_modes, pairs, slices=(), precision="tf32x3",
                 policy: int = TN_POLICY_AUTO):
        prec = PRECISIONS[precision] if isinstance(precision, str) else int(precision)
        self.handle = tn_plan(tensors, extents, open_modes, pairs, slices, prec)
        self.n_tensors = len(tensors)
        self.pairs = [(int(a), int(b)) for a, b in pairs]
        self.out_shape = tuple(int(extents[x]) for x in open_modes)
        # entries of every leaf (all its modes) and of the result
        self.leaf_sizes = [_prod(int(extents[x]) for x in t) for t in tensors]
        self.out_size = _prod(self.out_shape)
        self._ws = None
        if policy != TN_POLICY_AUTO:
            tn_plan_set_policy(self.handle, policy)

    @classmethod
    def from_network(cls, net, tree, slices=(), precision="tf32x3", policy=TN_POLICY_AUTO):
        return cls(net.tensors, net.extents, net.open_modes, tree, slices, precision, policy)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            tn_plan_destroy(h)
            self.handle = None

    flops = property(lambda self: tn_plan_flops(self.handle))
    peak = property(lambda self: tn_plan_peak(self.handle))
    num_slices = property(lambda self: tn_plan_num_slices(self.handle))
    num_steps = property(lambda self: tn_plan_num_steps(self.handle))
    workspace_bytes = property(lambda self: tn_plan_workspace_bytes(self.handle))

    def mode_order(self, tensor_id: int):
        return tn_plan_mode_order(self.handle, tensor_id)

    def node_mnk(self, step: int):
        return tn_plan_node_mnk(self.handle, step)

    def node_class(self, step: int) -> int:
        return tn_plan_node_class(self.handle, step)

    def set_policy(self, policy: int) -> None:
        tn_plan_set_policy(self.handle, policy)
        self._ws = None

    def set_three_products(self, enable: bool) -> None:
        tn_plan_set_three_products(self.handle, enable)
        self._ws = None

    def set_hoisting(self, enable: bool) -> None:
        tn_plan_set_hoisting(self.handle, enable)
        self._ws = None

    def set_fusion(self, enable: bool) -> None:
        tn_plan_set_fusion(self.handle, enable)
        self._ws = None

    def set_cta_pairs(self, enable: bool) -> None:
        tn_plan_set_cta_pairs(self.handle, enable)
        self._ws = None

    def set_promotion_chunk(self, chunk_k: int) -> None:
        tn_plan_set_promotion_chunk(self.handle, chunk_k)
        self._ws = None

    def bind_workspace(self, device=None):
        """Allocate the workspace with torch on ``device`` and bind it."""
        import torch
        nbytes = max(self.workspace_bytes, 256)
        self._ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        ptr = self._ws.data_ptr()
        aligned = (ptr + 255) // 256 * 256
        tn_plan_set_workspace(self.handle, aligned, nbytes)
        return self._ws

    def execute(self, leaves, out, stream=None) -> None:
        """Contract device leaves (complex64, contiguous, caller's order) into
        ``out`` (complex64, open-mode order).  Asynchronous on ``stream``
        (default: torch's current stream)."""
        import torch
        _check_buffers(self, leaves, out, True, "execute")
        if self._ws is None:
            self.bind_workspace(out.device)
        if stream is None:
            stream = torch.cuda.current_stream(out.device)
        sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        tn_execute(self.handle, [t.data_ptr() for t in leaves], out.data_ptr(), sp)

    def execute_slices(self, leaves, out, first: int, step: int, stream=None) -> None:
        """Sum of slices first, first + step, ... into ``out`` (see
        tn_execute_slices); with shard_slices this splits a sliced
        contraction over processes."""
        import torch
        _check_buffers(self, leaves, out, True, "execute_slices")
        if self._ws is None:
            self.bind_workspace(out.device)
        if stream is None:
            stream = torch.cuda.current_stream(out.device)
        sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        tn_execute_slices(self.handle, [t.data_ptr() for t in leaves], out.data_ptr(), sp,
                          first, step)

    def execute_host(self, host_leaves, host_out, dev_leaves, dev_out, stream=None) -> None:
        """End-to-end call with host buffers (tn_execute_host): the host
        leaves (pinned: one gather kernel; pageable: one copy each) into
        ``dev_leaves``, the contraction into ``dev_out``, the result into
        ``host_out``; then waits for the stream."""
        import torch
        _check_buffers(self, host_leaves, host_out, False, "execute_host")
        _check_buffers(self, dev_leaves, dev_out, True, "execute_host")
        if self._ws is None:
            self.bind_workspace(dev_out.device)
        if stream is None:
            stream = torch.cuda.current_stream(dev_out.device)
        sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        tn_execute_host(self.handle, [t.data_ptr() for t in host_leaves], host_out.data_ptr(),
                        [t.data_ptr() for t in dev_leaves], dev_out.data_ptr(), sp)
        stream.synchronize()

    def prepare_host(self, host_leaves, host_out, dev_leaves, dev_out, stream=None) -> "HostCall":
        """The same call as execute_host for buffers fixed in advance:
        checked and turned into pointer arrays once, so that each call of
        the returned object costs only tn_execute_host and the wait."""
        return HostCall(self, host_leaves, host_out, dev_leaves, dev_out, stream)

    def execute_prefix(self, leaves, out, step: int, stream=None) -> None:
        """Slice 0's launches up to the one computing ``step`` (see
        tn_execute_prefix); then ``gather`` reads that step's operands and
        output."""
        import torch
        _check_buffers(self, leaves, out, True, "execute_prefix")
        if self._ws is None:
            self.bind_workspace(out.device)
        if stream is None:
            stream = torch.cuda.current_stream(out.device)
        sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        tn_execute_prefix(self.handle, [t.data_ptr() for t in leaves], out.data_ptr(), step, sp)

    def gather(self, tensor_id: int, idx, stream=None):
        """Entries ``idx`` (an int64 CUDA tensor of logical row-major
        indices in the tensor's lifetime order) of tensor ``tensor_id`` as a
        complex64 CUDA tensor (tn_plan_tensor_gather)."""
        import torch
        if idx.dtype != torch.int64 or not idx.is_cuda or not idx.is_contiguous():
            raise ValueError("idx must be a contiguous int64 CUDA tensor")
        dst = torch.empty(idx.numel(), dtype=torch.complex64, device=idx.device)
        if stream is None:
            stream = torch.cuda.current_stream(idx.device)
        sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        tn_plan_tensor_gather(self.handle, tensor_id, idx.data_ptr(), idx.numel(), dst.data_ptr(), sp)
        return dst

    def check(self) -> None:
        tn_plan_check(self.handle)

    @property
    def launches(self) -> int:
        return tn_plan_launches(self.handle)

    def set_profiling(self, enable: bool) -> None:
        tn_plan_set_profiling(self.handle, enable)

    def profile(self):
        return tn_plan_profile_read(self.handle)


class HostCall:
    """A prepared tn_execute_host call (Plan.prepare_host): the buffers are
    checked once and held, their pointers kept in C arrays; calling the
    object runs leaves in, contraction, result out and waits for the
    stream.  The buffers must keep their storage while the object is used."""

    def __init__(self, plan: Plan, host_leaves, host_out, dev_leaves, dev_out, stream=None):
        import torch
        _check_buffers(plan, host_leaves, host_out, False, "prepare_host")
        _check_buffers(plan, dev_leaves, dev_out, True, "prepare_host")
        if plan._ws is None:
            plan.bind_workspace(dev_out.device)
        self.plan = plan
        self.buffers = (list(host_leaves), host_out, list(dev_leaves), dev_out)   # held alive
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev_out.device)
        self._sp = self.stream.cuda_stream if hasattr(self.stream, "cuda_stream") else int(self.stream)
        self._h = (_P * max(len(host_leaves), 1))(*[t.data_ptr() for t in host_leaves])
        self._d = (_P * max(len(dev_leaves), 1))(*[t.data_ptr() for t in dev_leaves])
        self._ho, self._do = host_out.data_ptr(), dev_out.data_ptr()
        self._fn = lib().tn_execute_host

    def __call__(self) -> None:
        _check(self._fn(self.plan.handle, self._h, self._ho, self._d, self._do, self._sp),
               self.plan.handle)
        self.stream.synchronize()
