"""Python binding of the C ABI in include/cc_dp.h (argument marshalling only).

Every function has the name of the C entry point it calls.  Pointer
arguments accept ``torch.Tensor`` (their ``data_ptr()``) or plain integers;
``stream`` accepts a ``torch.cuda.Stream``, a raw ``cudaStream_t`` integer,
or ``None`` for torch's current stream.  A non-OK status raises
:class:`CCError` carrying the status and the library's one-line reason.

There is no fallback: if ``libcc_dp.so`` has not been built, every call
raises.  Build it with ``python -c "import __graft_entry__ as g; g.build()"``
or ``python gradient_reduce_optimizer_gb300/build.py``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "libcc_dp.so")

CC_MAX_R = 16
CC_PAD_ELEMS = 8
CC_NOALLOC_SCRATCH_ELEMS = 16 * 1024 * 1024   # fixed scratch of the allocation-free entry point
CC_ARITH_FAST = 1                             # opt-in fast arithmetic of the bucket kernels
CC_ENGINE_BULK_COPY = 2                       # CTA budgets on the TMA bulk-copy engine
CC_TUNE_MAX_CANDIDATES = 64                   # bucket caps one tuning call may try
CC_OK = 0
CC_ERR_INVALID = -1
CC_ERR_ALIAS = -2
CC_ERR_MISALIGNED = -3
CC_ERR_CUDA = -4
CC_ERR_UNSUPPORTED = -5
CC_ERR_CAPACITY = -6

_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_f = ctypes.c_float
_i = ctypes.c_int


class CCError(RuntimeError):
    def __init__(self, status: int, func: str, reason: str):
        self.status = status
        self.func = func
        self.reason = reason
        super().__init__(f"{func}: {status_name(status)}: {reason}")


class cc_overlap_cfg(ctypes.Structure):
    _fields_ = [
        ("grads", _vp), ("acc", _vp), ("master", _vp), ("m", _vp), ("v", _vp),
        ("params_out", _vp), ("n", _sz), ("R", _i),
        ("bucket_begin", _vp), ("bucket_end", _vp),
        ("bucket_ready_layer", _vp), ("num_buckets", _i),
        ("lr", _f), ("beta1", _f), ("beta2", _f), ("eps", _f),
        ("weight_decay", _f), ("step", _i), ("grad_scale", _f),
        ("num_layers", _i), ("gemms_per_layer", _i),
        ("gemm_m", _i), ("gemm_n", _i), ("gemm_k", _i),
        ("gemm_a", _vp), ("gemm_b", _vp), ("gemm_c", _vp),
        ("warmup", _i), ("iters", _i), ("max_ctas", _i),
        ("stream_priority", _i), ("comm_sms", _i), ("budget_buckets", _i),
        ("gemm_algo", _i), ("arith_flags", ctypes.c_uint),
    ]


class cc_overlap_result(ctypes.Structure):
    _fields_ = [
        ("t_bwd_ms", _f), ("t_comm_ms", _f), ("t_step_overlap_ms", _f),
        ("t_step_seq_ms", _f), ("exposed_ms", _f), ("exposed_bound_ms", _f),
        ("num_buckets", _i), ("comm_sms", _i), ("compute_sms", _i),
        ("gemm_algos", _i), ("t_overlap_ms", _f), ("overlap_eff", _f),
    ]


class cc_tune_cfg(ctypes.Structure):
    _fields_ = [("overlap", cc_overlap_cfg), ("numel", _vp), ("layer_of", _vp),
                ("num_tensors", _i), ("candidates", _vp), ("num_candidates", _i),
                ("rank", _i)]


class cc_tune_result(ctypes.Structure):
    _fields_ = [("best", _i), ("best_bucket_bytes", _sz), ("num_candidates", _i)]


class cc_tp_cfg(ctypes.Structure):
    _fields_ = [
        ("R", _i), ("m", _i), ("n", _i), ("k", _i), ("chunks", _i),
        ("x", _vp), ("w", _vp), ("partials", _vp), ("out", _vp),
        ("warmup", _i), ("iters", _i), ("stream_priority", _i),
    ]


class cc_tp_result(ctypes.Structure):
    _fields_ = [("t_gemm_ms", _f), ("t_allreduce_ms", _f),
                ("t_sequential_ms", _f), ("t_overlap_ms", _f)]


_SIGNATURES = {
    "cc_status_string": ([_i], ctypes.c_char_p),
    "cc_last_error": ([], ctypes.c_char_p),
    "cc_fused_dp_step": ([_vp, _vp, _vp, _vp, _vp, _sz, _i, _sz, _f, _f, _f,
                          _f, _f, _i, _f, _i, _vp], _i),
    "cc_accumulate_local": ([_vp, _vp, _sz, _i, _i, _vp], _i),
    "cc_fused_dp_step_accum": ([_vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _sz,
                                _f, _f, _f, _f, _f, _i, _f, _i, _vp], _i),
    "cc_fused_dp_bucket": ([_vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _sz, _sz,
                            _f, _f, _f, _f, _f, _i, _f, _i, _vp], _i),
    "cc_fused_dp_shard": ([_vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _sz, _sz, _sz,
                           _f, _f, _f, _f, _f, _i, _f, _vp], _i),
    "cc_plan_buckets": ([_vp, _i, _sz, _vp, _vp, _vp, _i, _vp, _vp], _i),
    "cc_bucket_ready_layers": ([_vp, _vp, _vp, _i, _vp, _vp, _i, _vp], _i),
    "cc_overlap_bench": ([ctypes.POINTER(cc_overlap_cfg),
                          ctypes.POINTER(cc_overlap_result)], _i),
    "cc_tune_bucket_bytes": ([ctypes.POINTER(cc_tune_cfg), ctypes.POINTER(cc_overlap_result),
                              ctypes.POINTER(cc_tune_result)], _i),
    "cc_l2_flush": ([_vp, _sz, _vp], _i),
    "cc_device_status": ([ctypes.POINTER(ctypes.c_uint), _i], _i),
    "cc_unfused_dp_step": ([_vp, _vp, _vp, _vp, _vp, _vp, _sz, _sz, _i, _sz,
                            _f, _f, _f, _f, _f, _i, _f, _vp], _i),
    "cc_unfused_dp_step_noalloc": ([_vp, _vp, _vp, _vp, _vp, _sz, _i, _sz, _f, _f,
                                    _f, _f, _f, _i, _f, _vp], _i),
    "cc_tp_allreduce": ([_vp, _vp, _sz, _i, _vp], _i),
    "cc_fused_dp_bucket_ex": ([_vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _sz, _sz,
                               _f, _f, _f, _f, _f, _i, _f, _i, ctypes.c_uint, _vp], _i),
    "cc_shard_plan": ([_vp, _vp, _i, _i, _vp, _vp, _vp, _vp], _i),
    "cc_fused_dp_rank_step": ([_vp, _vp, _vp, _vp, _vp, _sz, _i, _f, _f, _f, _f, _f,
                               _i, _f, _vp], _i),
    "cc_tp_matmul_allreduce": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp], _i),
    "cc_tp_matmul_allreduce_ex": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _i, _vp],
                                  _i),
    "cc_tp_matmul_allreduce_workspace": ([_i, _i, _i, _i, _i, ctypes.POINTER(_sz)], _i),
    "cc_inject_bulk_stall": ([ctypes.c_longlong, ctypes.c_uint], _i),
    "cc_inject_launch_failure": ([_i], _i),
    "cc_tp_overlap_bench": ([ctypes.POINTER(cc_tp_cfg), ctypes.POINTER(cc_tp_result)], _i),
}

_LIB: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(
                f"{LIBRARY} is missing: the CUDA library must be built "
                "(python gradient_reduce_optimizer_gb300/build.py); "
                "there is no fallback path")
        L = ctypes.CDLL(LIBRARY)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = L
    return _LIB


def status_name(status: int) -> str:
    return lib().cc_status_string(status).decode()


def cc_status_string(status: int) -> str:
    return status_name(status)


def cc_last_error() -> str:
    return lib().cc_last_error().decode()


def _check(status: int, func: str) -> None:
    if status != CC_OK:
        raise CCError(status, func, cc_last_error())


def _addr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _addr_array(xs) -> Optional[ctypes.Array]:
    if xs is None:
        return None
    return (_vp * max(1, len(xs)))(*[_addr(x) for x in xs])


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def cc_fused_dp_step(grads, master, m, v, params_out, n: int, R: int,
                     bucket_bytes: int, lr: float, beta1: float, beta2: float,
                     eps: float, weight_decay: float, step: int,
                     grad_scale: float, accum_k: int = 1, stream=None) -> None:
    _check(lib().cc_fused_dp_step(
        _addr_array(grads), _addr(master), _addr(m), _addr(v),
        _addr_array(params_out), n, R, bucket_bytes, lr, beta1, beta2, eps,
        weight_decay, step, grad_scale, accum_k, _stream(stream)),
        "cc_fused_dp_step")


def cc_fused_dp_step_accum(grads, acc, master, m, v, params_out, n: int,
                           R: int, bucket_bytes: int, lr: float, beta1: float,
                           beta2: float, eps: float, weight_decay: float,
                           step: int, grad_scale: float, accum_k: int,
                           stream=None) -> None:
    _check(lib().cc_fused_dp_step_accum(
        _addr_array(grads), _addr_array(acc), _addr(master), _addr(m),
        _addr(v), _addr_array(params_out), n, R, bucket_bytes, lr, beta1,
        beta2, eps, weight_decay, step, grad_scale, accum_k, _stream(stream)),
        "cc_fused_dp_step_accum")


def cc_fused_dp_bucket(grads, acc, master, m, v, params_out, n: int, R: int,
                       begin: int, end: int, lr: float, beta1: float,
                       beta2: float, eps: float, weight_decay: float,
                       step: int, grad_scale: float, max_ctas: int = 0,
                       stream=None) -> None:
    _check(lib().cc_fused_dp_bucket(
        _addr_array(grads), _addr_array(acc), _addr(master), _addr(m),
        _addr(v), _addr_array(params_out), n, R, begin, end, lr, beta1, beta2,
        eps, weight_decay, step, grad_scale, max_ctas, _stream(stream)),
        "cc_fused_dp_bucket")


def cc_fused_dp_bucket_ex(grads, acc, master, m, v, params_out, n: int, R: int,
                          begin: int, end: int, lr: float, beta1: float,
                          beta2: float, eps: float, weight_decay: float,
                          step: int, grad_scale: float, max_ctas: int = 0,
                          arith_flags: int = 0, stream=None) -> None:
    _check(lib().cc_fused_dp_bucket_ex(
        _addr_array(grads), _addr_array(acc), _addr(master), _addr(m),
        _addr(v), _addr_array(params_out), n, R, begin, end, lr, beta1, beta2,
        eps, weight_decay, step, grad_scale, max_ctas, arith_flags, _stream(stream)),
        "cc_fused_dp_bucket_ex")


def cc_fused_dp_shard(grads, acc, master, m, v, params_out, n: int, R: int,
                      shard_begin: int, shard_end: int, bucket_bytes: int,
                      lr: float, beta1: float, beta2: float, eps: float,
                      weight_decay: float, step: int, grad_scale: float,
                      stream=None) -> None:
    _check(lib().cc_fused_dp_shard(
        _addr_array(grads), _addr_array(acc), _addr(master), _addr(m),
        _addr(v), _addr_array(params_out), n, R, shard_begin, shard_end,
        bucket_bytes, lr, beta1, beta2, eps, weight_decay, step, grad_scale,
        _stream(stream)), "cc_fused_dp_shard")


def cc_unfused_dp_step(grads, master, m, v, params_out, workspace,
                       workspace_bytes: int, n: int, R: int, bucket_bytes: int,
                       lr: float, beta1: float, beta2: float, eps: float,
                       weight_decay: float, step: int, grad_scale: float,
                       stream=None) -> None:
    _check(lib().cc_unfused_dp_step(
        _addr_array(grads), _addr(master), _addr(m), _addr(v),
        _addr_array(params_out), _addr(workspace), workspace_bytes, n, R,
        bucket_bytes, lr, beta1, beta2, eps, weight_decay, step, grad_scale,
        _stream(stream)), "cc_unfused_dp_step")


def cc_unfused_dp_step_noalloc(grads, master, m, v, params_out, n: int, R: int,
                               bucket_bytes: int, lr: float, beta1: float,
                               beta2: float, eps: float, weight_decay: float,
                               step: int, grad_scale: float, stream=None) -> None:
    """The unfused step for callers that cannot allocate: its scratch is a
    fixed 64 MiB array inside the library (buckets up to 16M elements)."""
    _check(lib().cc_unfused_dp_step_noalloc(
        _addr_array(grads), _addr(master), _addr(m), _addr(v),
        _addr_array(params_out), n, R, bucket_bytes, lr, beta1, beta2, eps,
        weight_decay, step, grad_scale, _stream(stream)),
        "cc_unfused_dp_step_noalloc")


def cc_accumulate_local(grads, acc, n: int, R: int, first: bool,
                        stream=None) -> None:
    _check(lib().cc_accumulate_local(_addr_array(grads), _addr_array(acc), n,
                                     R, int(bool(first)), _stream(stream)),
           "cc_accumulate_local")


def cc_plan_buckets(numel: Sequence[int], bucket_bytes: int
                    ) -> Tuple[List[int], List[Tuple[int, int]], int]:
    """Returns (offsets, [(begin, end), ...], n_padded)."""
    T = len(numel)
    c_numel = (_sz * T)(*numel)
    offsets = (_sz * T)()
    count = _i(0)
    n_pad = _sz(0)
    L = lib()
    st = L.cc_plan_buckets(c_numel, T, bucket_bytes, offsets, None, None, 0,
                           ctypes.byref(count), ctypes.byref(n_pad))
    if st not in (CC_OK, CC_ERR_CAPACITY):
        _check(st, "cc_plan_buckets")
    cap = count.value
    b = (_sz * max(1, cap))()
    e = (_sz * max(1, cap))()
    _check(L.cc_plan_buckets(c_numel, T, bucket_bytes, offsets, b, e, cap,
                             ctypes.byref(count), ctypes.byref(n_pad)),
           "cc_plan_buckets")
    return (list(offsets), [(b[i], e[i]) for i in range(count.value)],
            n_pad.value)


def cc_bucket_ready_layers(numel: Sequence[int], layer_of: Sequence[int],
                           offsets: Sequence[int],
                           buckets: Sequence[Tuple[int, int]]) -> List[int]:
    T, B = len(numel), len(buckets)
    out = (_i * max(1, B))()
    _check(lib().cc_bucket_ready_layers(
        (_sz * T)(*numel), (_i * T)(*layer_of), (_sz * T)(*offsets), T,
        (_sz * max(1, B))(*[b for b, _ in buckets]),
        (_sz * max(1, B))(*[e for _, e in buckets]), B, out),
        "cc_bucket_ready_layers")
    return list(out)[:B]


def _overlap_cfg(*, grads, master, m, v, params_out, n: int, R: int,
                 buckets: Sequence[Tuple[int, int]], ready_layers: Sequence[int], lr: float,
                 beta1: float, beta2: float, eps: float, weight_decay: float, step: int,
                 grad_scale: float, num_layers: int, gemms_per_layer: int, gemm_m: int,
                 gemm_n: int, gemm_k: int, gemm_a, gemm_b, gemm_c, warmup: int = 3,
                 iters: int = 20, max_ctas: int = 0, stream_priority: int = 0,
                 comm_sms: int = 0, budget_buckets: int = 0, gemm_algo: int = 0, acc=None,
                 arith_flags: int = 0):
    """A cc_overlap_cfg and the ctypes arrays it points into (keep both)."""
    B = len(buckets)
    keep = dict(
        g=_addr_array(grads), o=_addr_array(params_out),
        a=_addr_array(acc) if acc is not None else None,
        bb=(_sz * B)(*[b for b, _ in buckets]),
        be=(_sz * B)(*[e for _, e in buckets]),
        rl=(_i * B)(*ready_layers))
    cfg = cc_overlap_cfg(
        grads=ctypes.cast(keep["g"], _vp),
        acc=ctypes.cast(keep["a"], _vp) if keep["a"] is not None else None,
        master=_addr(master), m=_addr(m), v=_addr(v),
        params_out=ctypes.cast(keep["o"], _vp), n=n, R=R,
        bucket_begin=ctypes.cast(keep["bb"], _vp) if B else None,
        bucket_end=ctypes.cast(keep["be"], _vp) if B else None,
        bucket_ready_layer=ctypes.cast(keep["rl"], _vp) if B else None, num_buckets=B,
        lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay,
        step=step, grad_scale=grad_scale, num_layers=num_layers,
        gemms_per_layer=gemms_per_layer, gemm_m=gemm_m, gemm_n=gemm_n,
        gemm_k=gemm_k, gemm_a=_addr(gemm_a), gemm_b=_addr(gemm_b),
        gemm_c=_addr(gemm_c), warmup=warmup, iters=iters, max_ctas=max_ctas,
        stream_priority=stream_priority, comm_sms=comm_sms,
        budget_buckets=budget_buckets, gemm_algo=gemm_algo, arith_flags=arith_flags)
    return cfg, keep


def _result_dict(res) -> Dict[str, float]:
    return {name: getattr(res, name) for name, _ in res._fields_}


def cc_overlap_bench(**kw) -> Dict[str, float]:
    """The four timing arms of the bucketed step behind a proxy backward
    (keyword arguments: the cc_overlap_cfg fields; buckets as (begin, end)
    pairs and ready_layers)."""
    cfg, keep = _overlap_cfg(**kw)
    res = cc_overlap_result()
    _check(lib().cc_overlap_bench(ctypes.byref(cfg), ctypes.byref(res)),
           "cc_overlap_bench")
    return _result_dict(res)


def cc_tune_bucket_bytes(*, numel: Sequence[int], layer_of: Sequence[int],
                         candidates: Optional[Sequence[int]] = None, rank: int = -1,
                         **kw) -> Tuple[int, List[Dict[str, float]]]:
    """The measured best bucket cap: (cap in bytes, each candidate's overlap
    result).  Keyword arguments as cc_overlap_bench, without buckets and
    ready_layers; candidates None tries 1, 4, 25, 100 and 500 MiB."""
    cfg, keep = _overlap_cfg(buckets=[], ready_layers=[], **kw)
    T = len(numel)
    nm = (_sz * T)(*numel)
    lo = (_i * T)(*layer_of)
    cand = (_sz * len(candidates))(*candidates) if candidates is not None else None
    count = len(candidates) if candidates is not None else 5
    tcfg = cc_tune_cfg(overlap=cfg, numel=ctypes.cast(nm, _vp), layer_of=ctypes.cast(lo, _vp),
                       num_tensors=T, candidates=ctypes.cast(cand, _vp) if cand is not None else None,
                       num_candidates=len(candidates) if candidates is not None else 0,
                       rank=rank)
    results = (cc_overlap_result * max(count, 1))()
    out = cc_tune_result()
    _check(lib().cc_tune_bucket_bytes(ctypes.byref(tcfg), results, ctypes.byref(out)),
           "cc_tune_bucket_bytes")
    return out.best_bucket_bytes, [_result_dict(results[i]) for i in range(out.num_candidates)]


def cc_device_status(clear: bool = False) -> int:
    """The bulk engine's status word (0 = no wait ever ran out)."""
    st = ctypes.c_uint(0)
    _check(lib().cc_device_status(ctypes.byref(st), int(bool(clear))),
           "cc_device_status")
    return st.value


def cc_tp_allreduce(partials, out, n: int, R: int, stream=None) -> None:
    _check(lib().cc_tp_allreduce(_addr_array(partials), _addr_array(out), n, R,
                                 _stream(stream)), "cc_tp_allreduce")


def cc_tp_overlap_bench(*, R: int, m: int, n: int, k: int, chunks: int, x, w,
                        partials, out, warmup: int = 3, iters: int = 20,
                        stream_priority: int = 0) -> Dict[str, float]:
    keep = [_addr_array(a) for a in (x, w, partials, out)]
    cfg = cc_tp_cfg(R=R, m=m, n=n, k=k, chunks=chunks,
                    x=ctypes.cast(keep[0], _vp), w=ctypes.cast(keep[1], _vp),
                    partials=ctypes.cast(keep[2], _vp), out=ctypes.cast(keep[3], _vp),
                    warmup=warmup, iters=iters, stream_priority=stream_priority)
    res = cc_tp_result()
    _check(lib().cc_tp_overlap_bench(ctypes.byref(cfg), ctypes.byref(res)),
           "cc_tp_overlap_bench")
    return {name: getattr(res, name) for name, _ in res._fields_}


def cc_shard_plan(buckets: Sequence[Tuple[int, int]], world: int):
    """Shards of every bucket for `world` ranks: (shards, state_offsets,
    state_elems) with shards[b][q] = (begin, end) and state_offsets[b][q]
    the shard's place in rank q's state arrays."""
    B = len(buckets)
    bb = (_sz * max(1, B))(*[b for b, _ in buckets])
    be = (_sz * max(1, B))(*[e for _, e in buckets])
    sb = (_sz * max(1, B * world))()
    se = (_sz * max(1, B * world))()
    so = (_sz * max(1, B * world))()
    elems = (_sz * world)()
    _check(lib().cc_shard_plan(bb, be, B, world, sb, se, so, elems), "cc_shard_plan")
    shards = [[(sb[b * world + q], se[b * world + q]) for q in range(world)] for b in range(B)]
    offsets = [[so[b * world + q] for q in range(world)] for b in range(B)]
    return shards, offsets, list(elems)


def cc_fused_dp_rank_step(grad_slices, master, m, v, param_out, length: int, R: int, *,
                          lr: float, beta1: float, beta2: float, eps: float,
                          weight_decay: float, step: int, grad_scale: float,
                          stream=None) -> None:
    _check(lib().cc_fused_dp_rank_step(
        _addr_array(grad_slices), _addr(master), _addr(m), _addr(v), _addr(param_out),
        length, R, lr, beta1, beta2, eps, weight_decay, step, grad_scale, _stream(stream)),
        "cc_fused_dp_rank_step")


def cc_tp_matmul_allreduce(x, w, out, partials, m: int, n: int, k: int, R: int,
                           stream=None) -> None:
    """The fused tensor-parallel MatMul + AllReduce: x[r] bf16 m x k/R,
    w[r] bf16 n x k/R (K contiguous), out[r] bf16 m x n; partials None or
    [R] fp32 m x n (each rank's partial product, for checking)."""
    _check(lib().cc_tp_matmul_allreduce(
        _addr_array(x), _addr_array(w), _addr_array(out),
        _addr_array(partials) if partials is not None else None, m, n, k, R,
        _stream(stream)), "cc_tp_matmul_allreduce")


def cc_tp_matmul_allreduce_ex(x, w, out, partials, m: int, n: int, k: int, R: int,
                              workspace=None, workspace_bytes: int = 0, max_ctas: int = 0,
                              stream=None) -> None:
    """cc_tp_matmul_allreduce with a workspace (a device tensor, or None) in
    which the last wave's groups may be split, and a CTA budget (0: all)."""
    _check(lib().cc_tp_matmul_allreduce_ex(
        _addr_array(x), _addr_array(w), _addr_array(out),
        _addr_array(partials) if partials is not None else None, m, n, k, R,
        _addr(workspace) if workspace is not None else None, workspace_bytes, max_ctas,
        _stream(stream)), "cc_tp_matmul_allreduce_ex")


def cc_tp_matmul_allreduce_workspace(m: int, n: int, k: int, R: int, max_ctas: int = 0) -> int:
    """Workspace bytes cc_tp_matmul_allreduce_ex uses for this shape and CTA
    budget on the current device (0: it splits nothing)."""
    out = _sz(0)
    _check(lib().cc_tp_matmul_allreduce_workspace(m, n, k, R, max_ctas, ctypes.byref(out)),
           "cc_tp_matmul_allreduce_workspace")
    return out.value


def cc_inject_launch_failure(after_launches: int) -> None:
    """Arm (or with -1 disarm) a one-shot injected launch failure on this
    thread, for testing error propagation."""
    _check(lib().cc_inject_launch_failure(after_launches), "cc_inject_launch_failure")


def cc_inject_bulk_stall(tile: int, timeout_us: int = 20000) -> None:
    """Arm (or with -1 disarm) a one-shot skipped tile in the next bulk-engine
    launch on this thread, with its pipeline waits bounded by timeout_us."""
    _check(lib().cc_inject_bulk_stall(tile, timeout_us), "cc_inject_bulk_stall")


def cc_l2_flush(buf, nbytes: int, stream=None) -> None:
    _check(lib().cc_l2_flush(_addr(buf), nbytes, _stream(stream)),
           "cc_l2_flush")
