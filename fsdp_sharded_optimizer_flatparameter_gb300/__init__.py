"""Python binding of ``libzs.so``: the sharded mixed-precision AdamW step over a flat, padded buffer.

The functions here carry the C ABI's names (``include/zs.h``) and only
marshal arguments: torch tensors (or raw integer addresses) become pointers,
the current CUDA stream becomes the stream argument, and a negative status
becomes a :class:`ZsError`.  Every step of the method runs in the library's
CUDA kernels; there is no Python or CPU fallback.  When the shared library
is missing, importing this package raises an error that says how to build it.

Before a device call the binding checks that each tensor argument is a CUDA
tensor of the right element size holding at least the elements the call
will touch, because the C ABI receives bare pointers and cannot.
"""

import ctypes
import os

from ._lib import LIB_PATH, load_library

_lib = load_library()

ZS_OK = 0
ZS_ERR_INVALID = -1
ZS_ERR_CUDA = -2
ZS_ERR_OOM_HOST = -3
ZS_ERR_UNSUPPORTED = -5

ZS_STAGE_DP, ZS_STAGE_ZERO1, ZS_STAGE_ZERO2, ZS_STAGE_ZERO3 = 0, 1, 2, 3
ZS_RANK_FULL, ZS_SHARDED, ZS_RANK_BUCKET, ZS_RANK_UNIT = 0, 1, 2, 3
ZS_MAX_RANKS = 64
ZS_FUSED_AUTO, ZS_FUSED_LDG, ZS_FUSED_TMA = 0, 1, 2
ZS_BUCKETS_ONE_WALK, ZS_BUCKETS_PER_BUCKET = 0, 1
ZS_LAYOUT_FSDP1, ZS_LAYOUT_FSDP2 = 0, 1
ZS_DEVERR_NONE, ZS_DEVERR_PRODUCER_WAIT, ZS_DEVERR_CONSUMER_WAIT, ZS_DEVERR_SELFTEST = 0, 1, 2, 3
ZS_DEVERR_GATHER_WAIT = 4

c_i32, c_i64, c_f32, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
P_i64 = ctypes.POINTER(c_i64)
P_i32 = ctypes.POINTER(c_i32)


class ZsError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("zs status %d: %s" % (status, message))
        self.status = status


class zs_adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", c_f32), ("beta1", c_f32), ("beta2", c_f32), ("eps", c_f32), ("weight_decay", c_f32)]


def _sig(name, args, res=c_i32):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_sig("zs_plan_create", [c_i32, P_i32, P_i64, P_i32, c_i32, c_i32, c_i64, ctypes.POINTER(c_vp)])
_sig("zs_plan_destroy", [c_vp], None)
_sig("zs_plan_create_fsdp2", [c_i32, P_i32, P_i64, P_i32, c_i32, c_i32, c_i64, ctypes.POINTER(c_vp)])
_sig("zs_plan_layout", [c_vp, P_i32])
_sig("zs_plan_param_rows", [c_vp, c_i32, c_i32, P_i64, P_i64, P_i64, P_i64])
_sig("zs_plan_pad_ranges", [c_vp, P_i64, P_i64, c_i64, P_i64])
_sig("zs_fsdp2_chunk_cat", [c_vp, c_i32, c_vp, c_vp, c_vp])
_sig("zs_fsdp2_copy_out", [c_vp, c_i32, c_vp, c_vp, c_vp])
_sig("zs_plan_info", [c_vp, P_i64, P_i64, P_i64, P_i32, P_i32, P_i32, P_i32])
_sig("zs_plan_unit", [c_vp, c_i32, P_i64, P_i64, P_i64, P_i64])
_sig("zs_plan_bucket", [c_vp, c_i32, P_i32, P_i64, P_i64])
_sig("zs_plan_bucket_rank_slice", [c_vp, c_i32, c_i32, P_i64, P_i64])
_sig("zs_plan_param", [c_vp, c_i32, P_i32, P_i64, P_i64])
_sig("zs_plan_param_segment", [c_vp, c_i32, c_i32, P_i64, P_i64, P_i64])
_sig("zs_plan_memory_bytes", [c_vp, c_i32, P_i64])
_sig("zs_plan_comm_bytes", [c_vp, c_i32, c_i32, P_i64])
_sig("zs_adamw_scalars", [ctypes.POINTER(zs_adamw_hparams), c_i64, ctypes.POINTER(c_f32)])
_sig("zs_last_error", [], ctypes.c_char_p)
_sig("zs_accumulate_grad", [c_vp, c_vp, c_vp, c_f32, c_i32, c_vp])
_sig("zs_reduce_scatter_mean", [c_vp, c_i32, c_vp, c_i32, c_vp, c_i32, c_vp])
_sig("zs_adamw_shard_step", [c_vp, c_i32, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_i32,
                             ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp])
_sig("zs_all_gather", [c_vp, c_vp, c_i32, c_vp, c_vp])
_sig("zs_fused_step", [c_vp, c_i32, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp,
                       ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp])
_sig("zs_fused_step_accumulate", [c_vp, c_i32, c_vp, c_vp, c_i32, c_f32, c_vp, c_vp, c_vp, c_vp,
                                  ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp])
_sig("zs_fused_step_host", [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                            ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp, c_vp])
_sig("zs_zero3_gather_unit", [c_vp, c_i32, c_vp, c_vp, c_vp])
_sig("zs_zero3_rs_step_unit", [c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                               ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp])
_sig("zs_rank_shard_step", [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                            ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp])
_sig("zs_zero3_step", [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32,
                       ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp, c_vp])
_sig("zs_zero2_step_host", [c_vp, c_vp, c_vp, c_i64, c_vp, c_vp, c_vp, c_vp,
                            ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp, c_vp, c_vp, c_vp])
_sig("zs_checkpoint_save", [c_vp, ctypes.c_char_p, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp])
_sig("zs_checkpoint_load", [c_vp, ctypes.c_char_p, c_vp, c_vp, c_vp, c_vp, P_i64, c_vp])
_sig("zs_zero2_step_host_noalloc", [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.POINTER(zs_adamw_hparams), c_i64,
                                    c_vp, c_vp])
_sig("zs_all_reduce_mean", [c_vp, c_i32, c_vp, c_vp])
_sig("zs_dp_step", [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.POINTER(zs_adamw_hparams), c_i64, c_vp])
_sig("zs_fused_step_buckets", [c_vp, c_i32, P_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                               ctypes.POINTER(zs_adamw_hparams), c_i64, c_i32, c_vp, c_vp])
_sig("zs_set_fused_variant", [c_i32])
_sig("zs_set_dependent_launch", [c_i32])
_sig("zs_device_status", [ctypes.POINTER(ctypes.c_uint32), c_i32])
_sig("zs_selftest_wait_timeout", [c_i64, c_vp])

EXPORTED = [
    "zs_plan_create", "zs_plan_destroy", "zs_plan_info", "zs_plan_unit", "zs_plan_bucket",
    "zs_plan_bucket_rank_slice", "zs_plan_param", "zs_plan_param_segment", "zs_plan_memory_bytes",
    "zs_plan_comm_bytes", "zs_adamw_scalars", "zs_last_error", "zs_accumulate_grad",
    "zs_reduce_scatter_mean", "zs_adamw_shard_step", "zs_all_gather", "zs_fused_step",
    "zs_fused_step_host", "zs_zero3_gather_unit", "zs_zero3_rs_step_unit", "zs_set_fused_variant",
    "zs_device_status", "zs_selftest_wait_timeout", "zs_zero3_step", "zs_zero2_step_host",
    "zs_checkpoint_save", "zs_checkpoint_load", "zs_zero2_step_host_noalloc", "zs_all_reduce_mean",
    "zs_dp_step", "zs_plan_create_fsdp2", "zs_plan_layout", "zs_plan_param_rows", "zs_plan_pad_ranges",
    "zs_fsdp2_chunk_cat", "zs_fsdp2_copy_out", "zs_fused_step_buckets", "zs_set_dependent_launch",
    "zs_rank_shard_step", "zs_fused_step_accumulate",
]


def _check(status):
    if status != ZS_OK:
        raise ZsError(status, _lib.zs_last_error().decode())
    return status


def zs_last_error():
    return _lib.zs_last_error().decode()


# ------------------------------------------------------------------ plan

class Plan:
    """Owns a zs_plan_t.  Queries return plain Python integers."""

    def __init__(self, shapes, n_d, stage=ZS_STAGE_ZERO1, bucket_bytes=0, unit_of_param=None, layout=ZS_LAYOUT_FSDP1):
        self._h = None
        self._members = self._param_numel = None
        self._units, self._buckets = {}, {}      # query results, kept: the plan is immutable
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        shapes = [tuple(int(d) for d in s) for s in shapes]
        n = len(shapes)
        ndims = (c_i32 * max(n, 1))(*[len(s) for s in shapes])
        flat = [d for s in shapes for d in s]
        dims = (c_i64 * max(len(flat), 1))(*flat)
        units = None
        if unit_of_param is not None:
            units = (c_i32 * max(n, 1))(*[int(u) for u in unit_of_param])
        h = c_vp()
        create = _lib.zs_plan_create_fsdp2 if layout == ZS_LAYOUT_FSDP2 else _lib.zs_plan_create
        _check(create(n, ndims, dims, units, int(n_d), int(stage), int(bucket_bytes), ctypes.byref(h)))
        self._h = h
        info = self.info()
        self.numel, self.padded, self.shard_per_rank = info["numel"], info["padded"], info["shard_per_rank"]
        self.n_units, self.n_buckets, self.n_d, self.stage = (info["n_units"], info["n_buckets"],
                                                              info["n_d"], info["stage"])

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h is not None and self._h.value:
            _lib.zs_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self):
        a, b, c = c_i64(), c_i64(), c_i64()
        d, e, f, g = c_i32(), c_i32(), c_i32(), c_i32()
        _check(_lib.zs_plan_info(self._h, *(ctypes.byref(x) for x in (a, b, c, d, e, f, g))))
        return {"numel": a.value, "padded": b.value, "shard_per_rank": c.value, "n_units": d.value,
                "n_buckets": e.value, "n_d": f.value, "stage": g.value}

    def unit(self, u):
        u = int(u)
        got = self._units.get(u)
        if got is None:
            a, b, c, d = c_i64(), c_i64(), c_i64(), c_i64()
            _check(_lib.zs_plan_unit(self._h, u, *(ctypes.byref(x) for x in (a, b, c, d))))
            got = self._units[u] = (a.value, b.value, c.value, d.value)
        return {"base": got[0], "numel": got[1], "padded": got[2], "shard": got[3]}

    def unit_padded(self, u):
        """padded_u of unit u (the size of its ZS_RANK_UNIT buffers)."""
        u = int(u)
        got = self._units.get(u)
        return got[2] if got is not None else self.unit(u)["padded"]

    def bucket(self, b):
        b = int(b)
        got = self._buckets.get(b)
        if got is None:
            u, lo, hi = c_i32(), c_i64(), c_i64()
            _check(_lib.zs_plan_bucket(self._h, b, ctypes.byref(u), ctypes.byref(lo), ctypes.byref(hi)))
            got = self._buckets[b] = (u.value, lo.value, hi.value)
        return got

    def bucket_rank_slice(self, b, rank):
        lo, hi = c_i64(), c_i64()
        _check(_lib.zs_plan_bucket_rank_slice(self._h, int(b), int(rank), ctypes.byref(lo), ctypes.byref(hi)))
        return lo.value, hi.value

    def unit_local_offset(self, u):
        """Offset of unit u's shard in a rank's local layout (the units' shards back to back)."""
        return sum(self.unit(k)["shard"] for k in range(int(u)))

    def rank_bucket_part(self, rank, b):
        """Rank `rank`'s part of bucket b: (global begin, end, offset in the rank's local layout)."""
        lo, hi = self.bucket_rank_slice(b, rank)
        u = self.bucket(b)[0]
        ud = self.unit(u)
        s_lo = ud["base"] + int(rank) * ud["shard"]
        local = self.unit_local_offset(u) + (lo - s_lo) if hi > lo else self.unit_local_offset(u)
        return lo, hi, local

    def param(self, k):
        u, off, n = c_i32(), c_i64(), c_i64()
        _check(_lib.zs_plan_param(self._h, int(k), ctypes.byref(u), ctypes.byref(off), ctypes.byref(n)))
        return u.value, off.value, n.value

    def param_segment(self, k, rank):
        a, b, c = c_i64(), c_i64(), c_i64()
        _check(_lib.zs_plan_param_segment(self._h, int(k), int(rank), ctypes.byref(a), ctypes.byref(b),
                                          ctypes.byref(c)))
        return a.value, b.value, c.value

    def unit_members(self, u):
        """Indices of the parameters of unit u, in order (tabulated on first use; the plan is immutable)."""
        if self._members is None:
            members, numel = [[] for _ in range(self.n_units)], []
            for k in range(len(self.shapes)):
                unit, _, n = self.param(k)
                members[unit].append(k)
                numel.append(n)
            self._members, self._param_numel = members, numel
        return self._members[int(u)]

    def param_numel(self, k):
        if self._param_numel is None:
            self.unit_members(0)
        return self._param_numel[int(k)]

    def memory_bytes(self, stage=None):
        out = c_i64()
        _check(_lib.zs_plan_memory_bytes(self._h, self.stage if stage is None else int(stage), ctypes.byref(out)))
        return out.value

    def comm_bytes(self, stage=None, reshard_after_forward=True):
        out = c_i64()
        _check(_lib.zs_plan_comm_bytes(self._h, self.stage if stage is None else int(stage),
                                       1 if reshard_after_forward else 0, ctypes.byref(out)))
        return out.value

    def layout(self):
        out = c_i32()
        _check(_lib.zs_plan_layout(self._h, ctypes.byref(out)))
        return out.value

    def param_rows(self, k, rank):
        a, b, c, d = c_i64(), c_i64(), c_i64(), c_i64()
        _check(_lib.zs_plan_param_rows(self._h, int(k), int(rank), *(ctypes.byref(x) for x in (a, b, c, d))))
        return {"row_begin": a.value, "nrows": b.value, "rows_per_rank": c.value, "row_elems": d.value}

    def pad_ranges(self):
        count = c_i64()
        _check(_lib.zs_plan_pad_ranges(self._h, None, None, 0, ctypes.byref(count)))
        n = count.value
        begins, ends = (c_i64 * max(n, 1))(), (c_i64 * max(n, 1))()
        _check(_lib.zs_plan_pad_ranges(self._h, begins, ends, n, ctypes.byref(count)))
        return [(begins[i], ends[i]) for i in range(n)]


def zs_adamw_scalars(hp, step):
    out = (c_f32 * 8)()
    _check(_lib.zs_adamw_scalars(ctypes.byref(_hp(hp)), int(step), out))
    return list(out)


# ------------------------------------------------------------------ marshalling helpers

def _hp(hp):
    if isinstance(hp, zs_adamw_hparams):
        return hp
    return zs_adamw_hparams(float(hp["lr"]), float(hp["beta1"]), float(hp["beta2"]), float(hp["eps"]),
                            float(hp["weight_decay"]))


def _name(what):
    """An argument's name for a message: a string, or (name, index) formatted only when needed."""
    return what if isinstance(what, str) else "%s[%d]" % what


def _addr(x, min_elems=None, elem_size=None, what="buffer", device=True):
    """Address of a tensor (size-checked) or an integer address (unchecked).

    device=True: a CUDA tensor; "pinned_ok": a CUDA tensor or a pinned host tensor; False: any."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if device == "pinned_ok":
            if not (x.is_cuda or x.is_pinned()):
                raise ValueError("%s must be a CUDA tensor or pinned host memory" % _name(what))
        elif device and not x.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % _name(what))
        if not x.is_contiguous():
            raise ValueError("%s must be contiguous" % _name(what))
        if elem_size is not None and x.element_size() != elem_size:
            raise ValueError("%s must have %d-byte elements" % (_name(what), elem_size))
        if min_elems is not None and x.numel() < min_elems:
            raise ValueError("%s holds %d elements, the call touches %d" % (_name(what), x.numel(), min_elems))
        return x.data_ptr()
    raise TypeError("%s: expected a tensor or an integer address" % _name(what))


def _ptr_array(xs, min_elems, elem_size, what, device=True):
    if xs is None:
        return None
    vals = [_addr(x, min_elems, elem_size, (what, i), device) for i, x in enumerate(xs)]
    return (c_vp * max(len(vals), 1))(*vals)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _bf16_elems(plan, kind, bucket=-1, unit=0):
    if kind in (ZS_RANK_FULL, ZS_SHARDED):
        return plan.padded
    if kind == ZS_RANK_BUCKET:
        _, lo, hi = plan.bucket(bucket)
        return hi - lo
    if kind == ZS_RANK_UNIT:
        return plan.unit_padded(unit)
    raise ValueError("unknown buffer kind %r" % (kind,))


def _n_ptrs(kind, xs, n_d, what):
    want = 1 if kind == ZS_SHARDED else n_d
    if xs is not None and len(xs) != want:
        raise ValueError("%s: expected %d pointer(s), got %d" % (_name(what), want, len(xs)))


# ------------------------------------------------------------------ device operations

def zs_accumulate_grad(plan, acc, micro, scale, first, stream=None):
    _n_ptrs(ZS_RANK_FULL, acc, plan.n_d, "acc")
    _n_ptrs(ZS_RANK_FULL, micro, plan.n_d, "micro")
    return _check(_lib.zs_accumulate_grad(plan.handle, _ptr_array(acc, plan.padded, 2, "acc"),
                                          _ptr_array(micro, plan.padded, 2, "micro"), float(scale),
                                          1 if first else 0, _stream(stream)))


def zs_reduce_scatter_mean(plan, bucket, grads, grads_kind, out, out_kind, stream=None):
    _n_ptrs(grads_kind, grads, plan.n_d, "grads")
    _n_ptrs(out_kind, out, plan.n_d, "out")
    ng = _bf16_elems(plan, grads_kind, bucket)
    no = _bf16_elems(plan, out_kind, bucket)
    return _check(_lib.zs_reduce_scatter_mean(plan.handle, int(bucket), _ptr_array(grads, ng, 2, "grads"),
                                              int(grads_kind), _ptr_array(out, no, 2, "out"), int(out_kind),
                                              _stream(stream)))


def zs_adamw_shard_step(plan, rank, grad, grad_kind, master, m, v, params, params_kind, hp, step, stream=None):
    _n_ptrs(grad_kind, grad, plan.n_d, "grad")
    _n_ptrs(params_kind, params, plan.n_d, "params")
    n = plan.padded
    return _check(_lib.zs_adamw_shard_step(
        plan.handle, int(rank), _ptr_array(grad, n, 2, "grad"), int(grad_kind),
        _addr(master, n, 4, "master"), _addr(m, n, 4, "m"), _addr(v, n, 4, "v"),
        _ptr_array(params, n, 2, "params"), int(params_kind), ctypes.byref(_hp(hp)), int(step), _stream(stream)))


def zs_all_gather(plan, src, src_kind, replicas, stream=None):
    _n_ptrs(src_kind, src, plan.n_d, "src")
    _n_ptrs(ZS_RANK_FULL, replicas, plan.n_d, "replicas")
    n = plan.padded
    return _check(_lib.zs_all_gather(plan.handle, _ptr_array(src, n, 2, "src"), int(src_kind),
                                     _ptr_array(replicas, n, 2, "replicas"), _stream(stream)))


def zs_fused_step(plan, bucket, grads, grads_kind, master, m, v, replicas, hp, step, stream=None):
    _n_ptrs(grads_kind, grads, plan.n_d, "grads")
    _n_ptrs(ZS_RANK_FULL, replicas, plan.n_d, "replicas")
    n = plan.padded
    ng = _bf16_elems(plan, grads_kind, bucket)
    # gradients and replicas may be pinned host memory (read / written by the kernel over the host link)
    return _check(_lib.zs_fused_step(
        plan.handle, int(bucket), _ptr_array(grads, ng, 2, "grads", "pinned_ok"), int(grads_kind),
        _addr(master, n, 4, "master"), _addr(m, n, 4, "m"), _addr(v, n, 4, "v"),
        _ptr_array(replicas, n, 2, "replicas", "pinned_ok"), ctypes.byref(_hp(hp)), int(step), _stream(stream)))


def zs_fused_step_accumulate(plan, bucket, acc, micro, grads_kind, scale, master, m, v, replicas, hp, step,
                             stream=None):
    """zs_fused_step on the gradients bf16(acc[q] + micro[q] * scale): the last micro-batch's
    accumulation inside the step (acc and micro are only read)."""
    _n_ptrs(grads_kind, acc, plan.n_d, "acc")
    _n_ptrs(grads_kind, micro, plan.n_d, "micro")
    _n_ptrs(ZS_RANK_FULL, replicas, plan.n_d, "replicas")
    n = plan.padded
    ng = _bf16_elems(plan, grads_kind, bucket)
    return _check(_lib.zs_fused_step_accumulate(
        plan.handle, int(bucket), _ptr_array(acc, ng, 2, "acc", "pinned_ok"),
        _ptr_array(micro, ng, 2, "micro", "pinned_ok"), int(grads_kind), float(scale),
        _addr(master, n, 4, "master"), _addr(m, n, 4, "m"), _addr(v, n, 4, "v"),
        _ptr_array(replicas, n, 2, "replicas", "pinned_ok"), ctypes.byref(_hp(hp)), int(step), _stream(stream)))


def zs_fused_step_host(plan, host_grads, dev_grads, master, m, v, replicas, hp, step, host_replica0=None,
                       stream=None):
    _n_ptrs(ZS_RANK_FULL, host_grads, plan.n_d, "host_grads")
    _n_ptrs(ZS_RANK_FULL, dev_grads, plan.n_d, "dev_grads")
    n = plan.padded
    return _check(_lib.zs_fused_step_host(
        plan.handle, _ptr_array(host_grads, n, 2, "host_grads", device=False),
        _ptr_array(dev_grads, n, 2, "dev_grads"),
        _addr(master, n, 4, "master"), _addr(m, n, 4, "m"), _addr(v, n, 4, "v"),
        _ptr_array(replicas, n, 2, "replicas"), ctypes.byref(_hp(hp)), int(step),
        _addr(host_replica0, n, 2, "host_replica0", device=False), _stream(stream)))


def zs_zero3_gather_unit(plan, unit, shards, full, stream=None):
    _n_ptrs(ZS_RANK_UNIT, full, plan.n_d, "full")
    nu = plan.unit_padded(unit)
    return _check(_lib.zs_zero3_gather_unit(plan.handle, int(unit), _addr(shards, plan.padded, 2, "shards"),
                                            _ptr_array(full, nu, 2, "full"), _stream(stream)))


def zs_zero3_rs_step_unit(plan, unit, grads, master, m, v, shards, hp, step, stream=None):
    _n_ptrs(ZS_RANK_UNIT, grads, plan.n_d, "grads")
    n = plan.padded
    nu = plan.unit_padded(unit)
    return _check(_lib.zs_zero3_rs_step_unit(
        plan.handle, int(unit), _ptr_array(grads, nu, 2, "grads"),
        _addr(master, n, 4, "master"), _addr(m, n, 4, "m"), _addr(v, n, 4, "v"),
        _addr(shards, n, 2, "shards"), ctypes.byref(_hp(hp)), int(step), _stream(stream)))


def zs_rank_shard_step(plan, rank, bucket, slices, master, m, v, param_shard, hp, step, stream=None):
    """Rank `rank`'s local part of the step when every rank is its own process and GPU: slices are the
    N_d received gradient slices of its part of `bucket` (-1: of its whole shard); master, m, v and
    param_shard are the rank's own shard arrays in its local layout."""
    if bucket >= 0:
        lo, hi, _ = plan.rank_bucket_part(rank, bucket)
        n = hi - lo
    else:
        n = plan.shard_per_rank
    if len(slices) != plan.n_d:
        raise ValueError("slices must hold N_d = %d entries" % plan.n_d)
    ns = plan.shard_per_rank
    return _check(_lib.zs_rank_shard_step(
        plan.handle, int(rank), int(bucket), _ptr_array(slices, n, 2, "slices"),
        _addr(master, ns, 4, "master"), _addr(m, ns, 4, "m"), _addr(v, ns, 4, "v"),
        _addr(param_shard, ns, 2, "param_shard"), ctypes.byref(_hp(hp)), int(step), _stream(stream)))


def zs_zero3_step(plan, shards, master, m, v, unit_grads, pool, reshard_after_forward, hp, step,
                  main_stream=None, side_stream=None):
    """unit_grads: list (per unit) of N_d tensors; pool: list (per slot) of N_d tensors."""
    n, nd = plan.padded, plan.n_d
    if len(unit_grads) != plan.n_units:
        raise ValueError("unit_grads needs one list of N_d buffers per unit")
    biggest = max(plan.unit_padded(u) for u in range(plan.n_units))
    flat_g = []
    for u, per_rank in enumerate(unit_grads):
        _n_ptrs(ZS_RANK_UNIT, per_rank, nd, ("unit_grads", u))
        n_u = plan.unit_padded(u)
        flat_g += [_addr(x, n_u, 2, ("unit_grads", u)) for x in per_rank]
    flat_p = []
    for k, per_rank in enumerate(pool):
        _n_ptrs(ZS_RANK_UNIT, per_rank, nd, ("pool", k))
        flat_p += [_addr(x, biggest, 2, ("pool", k)) for x in per_rank]
    main = _stream(main_stream)
    side = main if side_stream is None else _stream(side_stream)
    return _check(_lib.zs_zero3_step(
        plan.handle, _addr(shards, n, 2, "shards"), _addr(master, n, 4, "master"), _addr(m, n, 4, "m"),
        _addr(v, n, 4, "v"), (c_vp * max(len(flat_g), 1))(*flat_g), (c_vp * max(len(flat_p), 1))(*flat_p),
        len(pool), 1 if reshard_after_forward else 0, ctypes.byref(_hp(hp)), int(step), main, side))


def zs_zero2_step_host(plan, host_grads, staging, master, m, v, replicas, hp, step, host_replica0=None,
                       stream=None, copy_stream=None, d2h_stream=None):
    """host_grads: N_d host tensors/addresses; staging: 2 lists of N_d device tensors (bucket-sized)."""
    n, nd = plan.padded, plan.n_d
    _n_ptrs(ZS_RANK_FULL, host_grads, nd, "host_grads")
    if len(staging) != 2:
        raise ValueError("staging needs 2 slots of N_d buffers")
    biggest = max(hi - lo for _, lo, hi in (plan.bucket(b) for b in range(plan.n_buckets)))
    flat_s = []
    for k, per_rank in enumerate(staging):
        _n_ptrs(ZS_RANK_BUCKET, per_rank, nd, ("staging", k))
        flat_s += [_addr(x, biggest, 2, ("staging", k)) for x in per_rank]
    main = _stream(stream)
    cp = _stream(copy_stream) if copy_stream is not None else main
    d2 = _stream(d2h_stream) if d2h_stream is not None else None
    return _check(_lib.zs_zero2_step_host(
        plan.handle, _ptr_array(host_grads, n, 2, "host_grads", device=False), (c_vp * len(flat_s))(*flat_s),
        biggest, _addr(master, n, 4, "master"), _addr(m, n, 4, "m"), _addr(v, n, 4, "v"),
        _ptr_array(replicas, n, 2, "replicas"), ctypes.byref(_hp(hp)), int(step),
        _addr(host_replica0, n, 2, "host_replica0", device=False), main, cp, d2))


def zs_checkpoint_save(plan, directory, shards, master, m, v, step, stream=None):
    n = plan.padded
    return _check(_lib.zs_checkpoint_save(plan.handle, os.fsencode(directory), _addr(shards, n, 2, "shards"),
                                          _addr(master, n, 4, "master"), _addr(m, n, 4, "m"), _addr(v, n, 4, "v"),
                                          int(step), _stream(stream)))


def zs_checkpoint_load(plan, directory, shards, master, m, v, stream=None):
    """Returns the saved step."""
    n = plan.padded
    step = c_i64()
    _check(_lib.zs_checkpoint_load(plan.handle, os.fsencode(directory), _addr(shards, n, 2, "shards"),
                                   _addr(master, n, 4, "master"), _addr(m, n, 4, "m"), _addr(v, n, 4, "v"),
                                   ctypes.byref(step), _stream(stream)))
    return step.value


def zs_zero2_step_host_noalloc(plan, host_grads, master, m, v, replicas, hp, step, host_replica0=None,
                               stream=None):
    """zs_zero2_step_host with the staging ring inside the library: allocates nothing."""
    n = plan.padded
    _n_ptrs(ZS_RANK_FULL, host_grads, plan.n_d, "host_grads")
    return _check(_lib.zs_zero2_step_host_noalloc(
        plan.handle, _ptr_array(host_grads, n, 2, "host_grads", device=False), _addr(master, n, 4, "master"),
        _addr(m, n, 4, "m"), _addr(v, n, 4, "v"), _ptr_array(replicas, n, 2, "replicas"), ctypes.byref(_hp(hp)),
        int(step), _addr(host_replica0, n, 2, "host_replica0", device=False), _stream(stream)))


def zs_all_reduce_mean(plan, bucket, grads, stream=None):
    _n_ptrs(ZS_RANK_FULL, grads, plan.n_d, "grads")
    return _check(_lib.zs_all_reduce_mean(plan.handle, int(bucket), _ptr_array(grads, plan.padded, 2, "grads"),
                                          _stream(stream)))


def zs_dp_step(plan, grads, master, m, v, replicas, hp, step, stream=None):
    """master, m, v, replicas: lists of N_d per-rank full buffers (each rank's own copy)."""
    n, nd = plan.padded, plan.n_d
    for name, xs in (("grads", grads), ("master", master), ("m", m), ("v", v), ("replicas", replicas)):
        _n_ptrs(ZS_RANK_FULL, xs, nd, name)
    return _check(_lib.zs_dp_step(
        plan.handle, _ptr_array(grads, n, 2, "grads"), _ptr_array(master, n, 4, "master"),
        _ptr_array(m, n, 4, "m"), _ptr_array(v, n, 4, "v"), _ptr_array(replicas, n, 2, "replicas"),
        ctypes.byref(_hp(hp)), int(step), _stream(stream)))


def _unit_params(plan, unit):
    if not 0 <= int(unit) < plan.n_units:
        raise ZsError(ZS_ERR_INVALID, "unit %d out of range" % int(unit))
    return plan.unit_members(unit)


def zs_fsdp2_chunk_cat(plan, unit, params, flat, stream=None):
    """params: the unit's parameters (bf16 tensors in their own layout), in order; flat: padded_u elements."""
    members = _unit_params(plan, unit)
    if len(params) != len(members):
        raise ValueError("expected %d parameters for unit %d" % (len(members), unit))
    ptrs = [_addr(x, plan.param_numel(k), 2, ("params", i)) for i, (x, k) in enumerate(zip(params, members))]
    return _check(_lib.zs_fsdp2_chunk_cat(plan.handle, int(unit), (c_vp * max(len(ptrs), 1))(*ptrs),
                                          _addr(flat, plan.unit_padded(unit), 2, "flat"), _stream(stream)))


def zs_fsdp2_copy_out(plan, unit, flat, params, stream=None):
    members = _unit_params(plan, unit)
    if len(params) != len(members):
        raise ValueError("expected %d parameters for unit %d" % (len(members), unit))
    ptrs = [_addr(x, plan.param_numel(k), 2, ("params", i)) for i, (x, k) in enumerate(zip(params, members))]
    return _check(_lib.zs_fsdp2_copy_out(plan.handle, int(unit), _addr(flat, plan.unit_padded(unit), 2, "flat"),
                                         (c_vp * max(len(ptrs), 1))(*ptrs), _stream(stream)))


def zs_fused_step_buckets(plan, buckets, grads, master, m, v, replicas, hp, step, launch_mode=None, stream=None,
                          side_stream=None):
    """buckets: bucket indices in stepping order.  launch_mode: ZS_BUCKETS_ONE_WALK (default:
    touching buckets merge, the ranges are walked in overlapping launches, runs under 2^16 elements
    share list launches) or ZS_BUCKETS_PER_BUCKET (the buckets walked one after another, no launch
    spanning two; odd positions on side_stream if given).  Gradients and replicas may be pinned host
    memory, as for zs_fused_step."""
    _n_ptrs(ZS_RANK_FULL, grads, plan.n_d, "grads")
    _n_ptrs(ZS_RANK_FULL, replicas, plan.n_d, "replicas")
    n = plan.padded
    ids = (c_i32 * max(len(buckets), 1))(*[int(b) for b in buckets])
    mode = ZS_BUCKETS_ONE_WALK if launch_mode is None else int(launch_mode)
    side = None if side_stream is None else _stream(side_stream)
    return _check(_lib.zs_fused_step_buckets(
        plan.handle, len(buckets), ids, _ptr_array(grads, n, 2, "grads", "pinned_ok"), _addr(master, n, 4, "master"),
        _addr(m, n, 4, "m"), _addr(v, n, 4, "v"), _ptr_array(replicas, n, 2, "replicas", "pinned_ok"),
        ctypes.byref(_hp(hp)), int(step), mode, _stream(stream), side))


def zs_set_fused_variant(variant):
    return _check(_lib.zs_set_fused_variant(int(variant)))


def zs_set_dependent_launch(enable):
    """Programmatic dependent launch for every kernel of the library (on by default)."""
    return _check(_lib.zs_set_dependent_launch(1 if enable else 0))


def zs_device_status(clear=False):
    code = ctypes.c_uint32()
    _check(_lib.zs_device_status(ctypes.byref(code), 1 if clear else 0))
    return code.value


def zs_selftest_wait_timeout(limit_cycles, stream=None):
    return _check(_lib.zs_selftest_wait_timeout(int(limit_cycles), _stream(stream)))


__all__ = ["Plan", "ZsError", "zs_adamw_hparams", "LIB_PATH"] + EXPORTED + [
    n for n in dir() if n.startswith("ZS_")]
