"""ctypes binding of libsp_gb300.so (argument marshalling only).

Every function here has the name of the C entry point it calls (include/
sp_gb300.h), takes torch tensors, passes their device pointers, sizes and
the current CUDA stream, and raises SPError on any non-OK status.  Nothing is
computed in Python: if the shared library is missing the import fails -- there
is no fallback.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsp_gb300.so")

SP_OK, SP_ERR_INVALID_ARG, SP_ERR_UNSUPPORTED, SP_ERR_WORKSPACE, SP_ERR_CUDA, \
    SP_ERR_DEVICE_TIMEOUT = range(6)
SP_BF16, SP_F32 = 0, 1
SP_ORDER_CONTIGUOUS, SP_ORDER_STRIPED = 0, 1

_ORDERS = {"contiguous": SP_ORDER_CONTIGUOUS, "striped": SP_ORDER_STRIPED}

EXPORTS = (
    "sp_status_string", "sp_ulysses_seq_to_head", "sp_ulysses_head_to_seq",
    "sp_ulysses_seq_to_head_qkv",
    "sp_segment_starts_workspace_bytes", "sp_segment_starts", "sp_blockwise_attn_workspace_bytes",
    "sp_blockwise_attn_split_workspace_bytes",
    "sp_blockwise_attn_fwd", "sp_blockwise_attn_step", "sp_blockwise_attn_fwd_noalloc",
    "sp_ring_block_step", "sp_ring_block_step_accumulate", "sp_query_block_attn_fwd",
    "sp_ring_block_step_bwd_workspace_bytes", "sp_ring_block_step_bwd",
    "sp_ulysses_ring_attn_workspace_bytes", "sp_ulysses_ring_attn_fwd",
    "sp_blockwise_attn_bwd_workspace_bytes", "sp_blockwise_attn_bwd", "sp_set_bwd_dq_reduction",
    "sp_attn_merge_partials",
    "sp_get_device_error", "sp_get_permute_error", "sp_permute_set_bulk_min_bytes",
    "sp_check_barrier_timeout",
    "sp_last_launch_count",
)


class SPError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {_lib.sp_status_string(status).decode()}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run sequence_parallelism_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "sp_status_string": (ctypes.c_char_p, [i]),
        "sp_ulysses_seq_to_head": (i, [vp, vp, i, i, i, i, i, i, vp]),
        "sp_ulysses_head_to_seq": (i, [vp, vp, i, i, i, i, i, i, vp]),
        "sp_ulysses_seq_to_head_qkv": (i, [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]),
        "sp_segment_starts_workspace_bytes": (sz, [i, i]),
        "sp_segment_starts": (i, [vp, vp, i, i, vp, sz, vp]),
        "sp_blockwise_attn_workspace_bytes": (sz, [i, i, i]),
        "sp_blockwise_attn_split_workspace_bytes": (sz, [i, i, i]),
        "sp_blockwise_attn_fwd": (i, [vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, vp, vp, sz,
                                      vp]),
        "sp_blockwise_attn_step": (i, [vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, vp, vp,
                                       sz, vp]),
        "sp_blockwise_attn_fwd_noalloc": (i, [vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, vp,
                                              vp]),
        "sp_ring_block_step_bwd_workspace_bytes": (sz, [i, i, i, i, i]),
        "sp_ring_block_step_bwd": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f,
                                       i, vp, vp, vp, vp, sz, vp]),
        "sp_ring_block_step": (i, [vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i, vp, vp, vp,
                                   sz, vp]),
        "sp_ring_block_step_accumulate": (i, [vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i,
                                              vp, vp, vp, sz, vp]),
        "sp_query_block_attn_fwd": (i, [vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, vp, vp,
                                        sz, vp]),
        "sp_ulysses_ring_attn_workspace_bytes": (sz, [i, i, i, i, i, i, i]),
        "sp_ulysses_ring_attn_fwd": (i, [vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, vp, vp,
                                         sz, vp]),
        "sp_blockwise_attn_bwd_workspace_bytes": (sz, [i, i, i, i, i]),
        "sp_blockwise_attn_bwd": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp,
                                      vp, vp, vp, sz, vp]),
        "sp_attn_merge_partials": (i, [vp, vp, i, i, i, i, i, i, vp, vp, vp]),
        "sp_get_device_error": (i, [vp, ctypes.POINTER(ctypes.c_int), vp]),
        "sp_get_permute_error": (i, [ctypes.POINTER(ctypes.c_int)]),
        "sp_permute_set_bulk_min_bytes": (sz, [sz]),
        "sp_set_bwd_dq_reduction": (i, [i]),
        "sp_check_barrier_timeout": (i, [vp, i, vp]),
        "sp_last_launch_count": (i, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return SP_BF16
    if t.dtype == torch.float32:
        return SP_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(fn, status):
    if status != SP_OK:
        raise SPError(fn, status)


def _dense(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def sp_status_string(status):
    return _lib.sp_status_string(status).decode()


def sp_last_launch_count():
    return _lib.sp_last_launch_count()


def sp_ulysses_seq_to_head(x, y, P, stream=None):
    """x [B][S][H][d] -> y [P][B][S][H/P][d]."""
    _dense(x, y)
    B, S, H, d = x.shape
    _check("sp_ulysses_seq_to_head", _lib.sp_ulysses_seq_to_head(
        _ptr(x), _ptr(y), B, S, H, d, P, _dtype(x), _stream(stream)))
    return y


def sp_ulysses_head_to_seq(y, x, P, stream=None):
    """y [P][B][S][H/P][d] -> x [B][S][H][d]."""
    _dense(x, y)
    B, S, H, d = x.shape
    _check("sp_ulysses_head_to_seq", _lib.sp_ulysses_head_to_seq(
        _ptr(y), _ptr(x), B, S, H, d, P, _dtype(x), _stream(stream)))
    return x


def sp_ulysses_seq_to_head_qkv(q, k, v, yq, yk, yv, P, stream=None):
    """q [B][S][Hq][d], k/v [B][S][Hkv][d] -> head-sharded yq, yk, yv (one launch)."""
    _dense(q, k, v, yq, yk, yv)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    _check("sp_ulysses_seq_to_head_qkv", _lib.sp_ulysses_seq_to_head_qkv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(yq), _ptr(yk), _ptr(yv), B, S, Hq, Hkv, d, P, _dtype(q),
        _stream(stream)))
    return yq, yk, yv


def sp_segment_starts_workspace_bytes(B, S):
    return _lib.sp_segment_starts_workspace_bytes(B, S)


def sp_segment_starts(position_ids, doc_start, workspace, stream=None):
    _dense(position_ids, doc_start, workspace)
    B, S = position_ids.shape
    _check("sp_segment_starts", _lib.sp_segment_starts(
        _ptr(position_ids), _ptr(doc_start), B, S, _ptr(workspace), workspace.numel()
        * workspace.element_size(), _stream(stream)))
    return doc_start


def sp_blockwise_attn_workspace_bytes(B, S, causal):
    return _lib.sp_blockwise_attn_workspace_bytes(B, S, int(bool(causal)))


def sp_blockwise_attn_split_workspace_bytes(B, S, causal):
    return _lib.sp_blockwise_attn_split_workspace_bytes(B, S, int(bool(causal)))


def sp_blockwise_attn_fwd(q, k, v, position_ids, P, order, scale, out, lse, workspace,
                          stream=None):
    _dense(q, k, v, position_ids, out, lse, workspace)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    _check("sp_blockwise_attn_fwd", _lib.sp_blockwise_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(position_ids), B, S, Hq, Hkv, d, P, _ORDERS[order],
        float(scale), _dtype(q), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def sp_blockwise_attn_fwd_noalloc(q, k, v, position_ids, P, order, scale, out, lse, stream=None):
    """sp_blockwise_attn_fwd with the library's built-in device scratch, for
    callers that cannot allocate device memory (no workspace argument)."""
    _dense(q, k, v, position_ids, out, lse)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    _check("sp_blockwise_attn_fwd_noalloc", _lib.sp_blockwise_attn_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(position_ids), B, S, Hq, Hkv, d, P, _ORDERS[order],
        float(scale), _dtype(q), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def sp_blockwise_attn_step(q, k, v, position_ids, P, order, step, scale, out, lse, workspace,
                           stream=None):
    _dense(q, k, v, position_ids, out, lse, workspace)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    _check("sp_blockwise_attn_step", _lib.sp_blockwise_attn_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(position_ids), B, S, Hq, Hkv, d, P, _ORDERS[order], step,
        float(scale), _dtype(q), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def sp_ring_block_step(q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, scale, out_blk,
                       lse_blk, workspace, stream=None):
    """One device's ring step: query block i against key/value block j
    (block tensors [B][S/P][H][d]; position_ids of the whole sequence)."""
    _dense(q_blk, k_blk, v_blk, position_ids, out_blk, lse_blk, workspace)
    B, Lb, Hq, d = q_blk.shape
    Hkv = k_blk.shape[2]
    if Lb * P != S or k_blk.shape[1] != Lb:
        raise ValueError("block tensors must hold S/P rows")
    _check("sp_ring_block_step", _lib.sp_ring_block_step(
        _ptr(q_blk), _ptr(k_blk), _ptr(v_blk), _ptr(position_ids), B, S, Hq, Hkv, d, P,
        _ORDERS[order], i, j, float(scale), _dtype(q_blk), _ptr(out_blk), _ptr(lse_blk),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out_blk, lse_blk


def sp_ring_block_step_accumulate(q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, scale,
                                  out_blk, lse_blk, workspace, stream=None):
    """sp_ring_block_step folded into the running result (out_blk, lse_blk),
    which it updates in place."""
    _dense(q_blk, k_blk, v_blk, position_ids, out_blk, lse_blk, workspace)
    if lse_blk is None:
        raise ValueError("the running lse is required")
    B, Lb, Hq, d = q_blk.shape
    Hkv = k_blk.shape[2]
    if Lb * P != S or k_blk.shape[1] != Lb:
        raise ValueError("block tensors must hold S/P rows")
    _check("sp_ring_block_step_accumulate", _lib.sp_ring_block_step_accumulate(
        _ptr(q_blk), _ptr(k_blk), _ptr(v_blk), _ptr(position_ids), B, S, Hq, Hkv, d, P,
        _ORDERS[order], i, j, float(scale), _dtype(q_blk), _ptr(out_blk), _ptr(lse_blk),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out_blk, lse_blk


def sp_ring_block_step_bwd_workspace_bytes(B, S, Hq, P, causal):
    return int(_lib.sp_ring_block_step_bwd_workspace_bytes(B, S, Hq, P, 1 if causal else 0))


def sp_ring_block_step_bwd(q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk, position_ids, S, P,
                           order, i, j, scale, dq_acc, dk_acc, dv_acc, workspace, stream=None):
    """Backward of one device's ring step: adds block pair (i, j)'s part of
    the gradients into the float32 accumulators dq_acc ([B][S/P][Hq][d]),
    dk_acc, dv_acc ([B][S/P][Hkv][d]); lse_blk is block i's forward lse."""
    _dense(q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk, position_ids, dq_acc, dk_acc, dv_acc,
           workspace)
    B, Lb, Hq, d = q_blk.shape
    Hkv = k_blk.shape[2]
    if Lb * P != S or k_blk.shape[1] != Lb:
        raise ValueError("block tensors must hold S/P rows")
    if any(t.dtype != torch.float32 for t in (dq_acc, dk_acc, dv_acc)):
        raise ValueError("the gradient accumulators are float32")
    _check("sp_ring_block_step_bwd", _lib.sp_ring_block_step_bwd(
        _ptr(q_blk), _ptr(k_blk), _ptr(v_blk), _ptr(out_blk), _ptr(dout_blk), _ptr(lse_blk),
        _ptr(position_ids), B, S, Hq, Hkv, d, P, _ORDERS[order], i, j, float(scale),
        _dtype(q_blk), _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dq_acc, dk_acc, dv_acc


def sp_query_block_attn_fwd(q_blk, k, v, position_ids, P, order, i, scale, out_blk, lse_blk,
                            workspace, stream=None):
    """Query block i (block tensor [B][S/P][Hq][d]) against the whole
    sequence's k, v ([B][S][Hkv][d]) in ring order."""
    _dense(q_blk, k, v, position_ids, out_blk, lse_blk, workspace)
    B, Lb, Hq, d = q_blk.shape
    S, Hkv = k.shape[1], k.shape[2]
    if Lb * P != S:
        raise ValueError("q_blk must hold S/P rows")
    _check("sp_query_block_attn_fwd", _lib.sp_query_block_attn_fwd(
        _ptr(q_blk), _ptr(k), _ptr(v), _ptr(position_ids), B, S, Hq, Hkv, d, P, _ORDERS[order],
        i, float(scale), _dtype(q_blk), _ptr(out_blk), _ptr(lse_blk), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out_blk, lse_blk


def sp_ulysses_ring_attn_workspace_bytes(B, S, Hq, Hkv, d, causal, dtype):
    return _lib.sp_ulysses_ring_attn_workspace_bytes(B, S, Hq, Hkv, d, int(bool(causal)), dtype)


def sp_ulysses_ring_attn_fwd(q, k, v, position_ids, P_u, P_r, order, scale, out, lse, workspace,
                             stream=None):
    """Ulysses (P_u head groups) + ring (P_r blocks) hybrid; lse in the
    head-sharded layout [P_u][B][Hq/P_u][S]."""
    _dense(q, k, v, position_ids, out, lse, workspace)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    _check("sp_ulysses_ring_attn_fwd", _lib.sp_ulysses_ring_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(position_ids), B, S, Hq, Hkv, d, P_u, P_r,
        _ORDERS[order], float(scale), _dtype(q), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, causal):
    return _lib.sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, int(bool(causal)))


def sp_blockwise_attn_bwd(q, k, v, out, dout, lse, position_ids, P, order, scale, dq, dk, dv,
                          workspace, stream=None):
    _dense(q, k, v, out, dout, lse, position_ids, dq, dk, dv, workspace)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    _check("sp_blockwise_attn_bwd", _lib.sp_blockwise_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(position_ids), B, S,
        Hq, Hkv, d, P, _ORDERS[order], float(scale), _dtype(q), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return dq, dk, dv


def sp_attn_merge_partials(outs, lses, out, lse, stream=None):
    """outs [P][B][S][H][d], lses [P][B][H][S] -> out [B][S][H][d], lse [B][H][S]."""
    _dense(outs, lses, out, lse)
    P, B, S, H, d = outs.shape
    _check("sp_attn_merge_partials", _lib.sp_attn_merge_partials(
        _ptr(outs), _ptr(lses), P, B, S, H, d, _dtype(outs), _ptr(out), _ptr(lse),
        _stream(stream)))
    return out, lse


def sp_get_device_error(workspace, stream=None):
    code = ctypes.c_int(0)
    st = _lib.sp_get_device_error(_ptr(workspace), ctypes.byref(code), _stream(stream))
    return st, code.value


def sp_get_permute_error():
    code = ctypes.c_int(0)
    st = _lib.sp_get_permute_error(ctypes.byref(code))
    return st, code.value


def sp_permute_set_bulk_min_bytes(min_bytes):
    return int(_lib.sp_permute_set_bulk_min_bytes(int(min_bytes)))


def sp_set_bwd_dq_reduction(on):
    return int(_lib.sp_set_bwd_dq_reduction(1 if on else 0))


def sp_check_barrier_timeout(workspace, timeout_us, stream=None):
    _dense(workspace)
    _check("sp_check_barrier_timeout", _lib.sp_check_barrier_timeout(
        _ptr(workspace), int(timeout_us), _stream(stream)))
