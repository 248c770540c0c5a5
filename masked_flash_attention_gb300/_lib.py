"""ctypes binding of libmfa_gb300.so (argument marshalling only).

Every function here mirrors an entry point of ``include/fa.h`` by name.  Torch
is used for device memory and streams: tensors are described to the library
as (pointer, dtype, shape, strides) and every step of the attention runs in the
library's CUDA kernels.  There is no fallback: if the shared library is
missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import struct

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmfa_gb300.so")

# FA_ABI_VERSION of include/fa.h that the structures below describe
ABI_VERSION = 8

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_WORKSPACE = 3
FA_ERR_CUDA = 4
FA_ERR_DEVICE_TIMEOUT = 5
FA_ERR_DEVICE_BOUNDS = 6
FA_ERR_NO_DEVICE = 7
FA_ERR_DEVICE_VALUE = 8

FA_DTYPE_BF16, FA_DTYPE_F32, FA_DTYPE_I32, FA_DTYPE_F16 = 1, 2, 3, 4
FA_MASK_NONE, FA_MASK_DENSE, FA_MASK_TOPK = 0, 1, 2
FA_DEBUG_NO_SKIP = 0x1
FA_DEBUG_WITHHOLD = 0x2
FA_DEBUG_VALIDATE = 0x4
FA_PATH_DECODE, FA_PATH_PREFILL = 1, 2
FA_TILE_EMPTY, FA_TILE_FULL, FA_TILE_PARTIAL = 0, 1, 2

_DTYPES = {torch.bfloat16: FA_DTYPE_BF16, torch.float32: FA_DTYPE_F32, torch.int32: FA_DTYPE_I32,
           torch.float16: FA_DTYPE_F16}


class fa_tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class fa_mask(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("keep_window", ctypes.c_int32), ("t", fa_tensor)]


class fa_opts(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("max_seqlen_q", ctypes.c_int32),
                ("max_seqlen_k", ctypes.c_int32), ("debug_flags", ctypes.c_uint32),
                ("reserved", ctypes.c_int32), ("event_begin", ctypes.c_void_p),
                ("event_end", ctypes.c_void_p), ("alibi_slopes", ctypes.c_void_p),
                ("event_attn_end", ctypes.c_void_p)]


class fa_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("n_seq", ctypes.c_int32),
                ("n_heads_sched", ctypes.c_int32), ("n_row_tiles", ctypes.c_int32),
                ("rows_per_tile", ctypes.c_int32), ("keys_per_tile", ctypes.c_int32),
                ("n_k_tiles", ctypes.c_int32), ("n_splits", ctypes.c_int32),
                ("tiles_per_split", ctypes.c_int32), ("tail_units", ctypes.c_int32),
                ("n_items", ctypes.c_int64), ("off_counts", ctypes.c_size_t),
                ("off_tiles", ctypes.c_size_t), ("off_stats", ctypes.c_size_t),
                ("off_topk_e", ctypes.c_size_t), ("off_topk_list", ctypes.c_size_t),
                ("n_kernels", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_P = ctypes.POINTER
_ARGS = [_P(fa_tensor), _P(fa_tensor), _P(fa_tensor), _P(fa_tensor), _P(fa_tensor),
         _P(fa_tensor), _P(fa_tensor), _P(fa_tensor), _P(fa_mask), ctypes.c_int32,
         ctypes.c_int32, ctypes.c_float, ctypes.c_float, ctypes.c_int32, _P(fa_opts)]

# fa_fwd_kvcache / fa_fwd_kvcache_plan: q, k_cache, v_cache, k_new, v_new, out, lse,
# cu_seqlens_q, cache_seqlens, block_table, window_left, window_right, softcap,
# scale, causal, append, opts
_KV_ARGS = [_P(fa_tensor)] * 10 + [ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                   ctypes.c_int32, ctypes.c_int32, _P(fa_opts)]

# fa_bwd / fa_bwd_plan: q, k, v, out, lse, dout, dq, dk, dv, cu_seqlens_q,
# cu_seqlens_k, window_left, window_right, softcap, scale, causal, opts
_BWD_ARGS = [_P(fa_tensor)] * 11 + [ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_int32, _P(fa_opts)]

EXPORTS = ("fa_fwd", "fa_fwd_plan", "fa_fwd_workspace_size", "fa_fwd_kvcache", "fa_fwd_kvcache_plan",
           "fa_bwd", "fa_bwd_plan", "fa_fwd_noalloc", "fa_check_device_error", "fa_status_string",
           "fa_abi_version", "fa_fwd_debug_dump", "fa_debug_dump_bytes")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    missing = [name for name in EXPORTS if not hasattr(lib, name)]
    if missing:
        raise ImportError(f"{LIB_PATH} lacks {', '.join(missing)}: rebuild it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib.fa_fwd.argtypes = _ARGS
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_fwd_plan.argtypes = _ARGS + [_P(fa_plan)]
    lib.fa_fwd_plan.restype = ctypes.c_int
    lib.fa_fwd_workspace_size.argtypes = _ARGS + [_P(ctypes.c_size_t)]
    lib.fa_fwd_workspace_size.restype = ctypes.c_int
    lib.fa_fwd_kvcache.argtypes = _KV_ARGS
    lib.fa_fwd_kvcache.restype = ctypes.c_int
    lib.fa_fwd_kvcache_plan.argtypes = _KV_ARGS + [_P(fa_plan)]
    lib.fa_fwd_kvcache_plan.restype = ctypes.c_int
    lib.fa_bwd.argtypes = _BWD_ARGS
    lib.fa_bwd.restype = ctypes.c_int
    lib.fa_bwd_plan.argtypes = _BWD_ARGS + [_P(fa_plan)]
    lib.fa_bwd_plan.restype = ctypes.c_int
    lib.fa_fwd_noalloc.argtypes = _ARGS
    lib.fa_fwd_noalloc.restype = ctypes.c_int
    lib.fa_check_device_error.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _P(ctypes.c_uint32)]
    lib.fa_check_device_error.restype = ctypes.c_int
    lib.fa_status_string.argtypes = [ctypes.c_int]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_abi_version.argtypes = []
    lib.fa_abi_version.restype = ctypes.c_int
    lib.fa_fwd_debug_dump.argtypes = [_P(fa_tensor)] * 7 + [ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                                            ctypes.c_float, ctypes.c_int32, _P(fa_opts),
                                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                            ctypes.c_void_p, ctypes.c_size_t]
    lib.fa_fwd_debug_dump.restype = ctypes.c_int
    lib.fa_debug_dump_bytes.argtypes = [ctypes.c_int64]
    lib.fa_debug_dump_bytes.restype = ctypes.c_size_t
    # a library built from other headers would read these structures wrongly
    if lib.fa_abi_version() != ABI_VERSION:
        raise ImportError(f"{LIB_PATH} has ABI {lib.fa_abi_version()}, this binding describes ABI {ABI_VERSION}: "
                          "rebuild it with `python -c 'import __graft_entry__ as g; g.build()'`")
    return lib


lib = _load()


class FaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {lib.fa_status_string(status).decode()} (status {status})")


def fa_status_string(status: int) -> str:
    return lib.fa_status_string(int(status)).decode()


def fa_abi_version() -> int:
    return lib.fa_abi_version()


# fa_tensor's bytes: data pointer, dtype, ndim, shape[4], stride[4] (native
# byte order, no padding), packed in one call: the struct is built on every
# fa_fwd, so this keeps the host side of a call short
_TENSOR_BYTES = struct.Struct("=Qii4q4q")
assert _TENSOR_BYTES.size == ctypes.sizeof(fa_tensor)


def describe(t: torch.Tensor | None):
    """fa_tensor for a torch tensor (None -> None)."""
    if t is None:
        return None
    nd = t.dim()
    if nd > 4:
        raise ValueError("at most 4 dimensions")
    pad = (0,) * (4 - nd)
    # an empty tensor may have no storage: a dummy non-null pointer (never read)
    return fa_tensor.from_buffer_copy(_TENSOR_BYTES.pack(t.data_ptr() or 16, _DTYPES.get(t.dtype, 0), nd,
                                                         *t.shape, *pad, *t.stride(), *pad))


def _ref(x):
    return ctypes.byref(x) if x is not None else None


def _args(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask, zero_hold_states,
          keep_window, window_left, window_right, softcap, scale, causal, opts):
    m = None
    if mask is not None:
        m = fa_mask(FA_MASK_DENSE, 0, describe(mask))
    elif zero_hold_states is not None:
        m = fa_mask(FA_MASK_TOPK, int(keep_window), describe(zero_hold_states))
    descs = [describe(x) for x in (q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table)]
    keep = (descs, m, opts)  # keep the structs alive for the call
    args = [_ref(x) for x in descs] + [_ref(m), int(window_left), int(window_right),
                                       float(softcap), float(scale), int(bool(causal)),
                                       ctypes.byref(opts)]
    return args, keep


def _out_shapes(q, cu_seqlens_q, max_seqlen_q):
    if cu_seqlens_q is not None:
        return q.shape, (q.shape[1], q.shape[0])
    return q.shape, (q.shape[0], q.shape[2], q.shape[1])


def make_opts(stream=None, workspace=None, max_seqlen_q=0, max_seqlen_k=0, debug_flags=0,
              event_begin=None, event_end=None, alibi_slopes=None, event_attn_end=None):
    o = fa_opts()
    o.alibi_slopes = alibi_slopes.data_ptr() if alibi_slopes is not None else None
    o.event_begin = event_begin.cuda_event if event_begin is not None else None
    o.event_end = event_end.cuda_event if event_end is not None else None
    o.event_attn_end = event_attn_end.cuda_event if event_attn_end is not None else None
    o.stream = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    o.workspace = workspace.data_ptr() if workspace is not None else None
    o.workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    o.max_seqlen_q = int(max_seqlen_q or 0)
    o.max_seqlen_k = int(max_seqlen_k or 0)
    o.debug_flags = int(debug_flags)
    return o


def fa_fwd_plan(q, k, v, *, out=None, lse=None, cu_seqlens_q=None, cu_seqlens_k=None,
                block_table=None, mask=None, zero_hold_states=None, keep_window=0,
                window_left=-1, window_right=-1, softcap=0.0, scale=None, causal=False,
                max_seqlen_q=None, max_seqlen_k=None, debug_flags=0, stream=0, **_):
    """Host-only plan query; returns (status, plan dict).  ``out``/``lse`` may
    be omitted (a same-shaped stand-in descriptor is used)."""
    if out is None:
        out = q
    if lse is None:
        lse = torch.empty(_out_shapes(q, cu_seqlens_q, max_seqlen_q)[1], dtype=torch.float32,
                          device=q.device)
    opts = make_opts(stream=stream, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                     debug_flags=debug_flags)
    args, keep = _args(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask,
                       zero_hold_states, keep_window, window_left, window_right, softcap,
                       scale or 0.0, causal, opts)
    plan = fa_plan()
    rc = lib.fa_fwd_plan(*args, ctypes.byref(plan))
    return rc, plan.as_dict()


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """Zero-filled, 256-byte aligned device workspace (torch allocates it)."""
    return torch.zeros(max(256, int(nbytes)), dtype=torch.uint8, device=device)


def _alibi(slopes, q):
    """Checked ALiBi slopes: a contiguous fp32 CUDA tensor with one value per
    query head, on q's device (or None)."""
    if slopes is None:
        return None
    if (not isinstance(slopes, torch.Tensor) or slopes.dtype != torch.float32 or not slopes.is_cuda
            or slopes.device != q.device or slopes.dim() != 1 or slopes.numel() != q.shape[-2]
            or not slopes.is_contiguous()):
        raise FaError(FA_ERR_INVALID_ARG, "alibi_slopes (fp32 CUDA tensor [Hq] on q's device)")
    return slopes


def fa_fwd(q, k, v, *, out=None, lse=None, cu_seqlens_q=None, cu_seqlens_k=None,
           block_table=None, mask=None, zero_hold_states=None, keep_window=0, window_left=-1,
           window_right=-1, softcap=0.0, scale=None, causal=False, max_seqlen_q=None,
           max_seqlen_k=None, workspace=None, stream=None, debug_flags=0, event_begin=None,
           event_end=None, alibi_slopes=None, event_attn_end=None, **_):
    """Masked attention forward on the GPU through the C ABI.  Returns
    ``(out, lse, workspace)``; ``out``/``lse``/``workspace`` are allocated with
    torch when not given.  ``alibi_slopes``: optional fp32 CUDA tensor [Hq].
    Raises FaError on a non-zero status."""
    if not q.is_cuda:
        raise FaError(FA_ERR_INVALID_ARG, "fa_fwd (tensors must be CUDA tensors)")
    oshape, lshape = _out_shapes(q, cu_seqlens_q, max_seqlen_q)
    if out is None:
        out = torch.empty(oshape, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(lshape, dtype=torch.float32, device=q.device)
    alibi_slopes = _alibi(alibi_slopes, q)
    opts = make_opts(stream=stream, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                     debug_flags=debug_flags, event_begin=event_begin, event_end=event_end,
                     alibi_slopes=alibi_slopes, event_attn_end=event_attn_end)
    args, keep = _args(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask,
                       zero_hold_states, keep_window, window_left, window_right, softcap,
                       scale or 0.0, causal, opts)
    if workspace is None:
        nbytes = ctypes.c_size_t(0)
        rc = lib.fa_fwd_workspace_size(*args, ctypes.byref(nbytes))
        if rc != FA_OK:
            raise FaError(rc, "fa_fwd_workspace_size")
        workspace = alloc_workspace(nbytes.value, q.device)
    opts.workspace = workspace.data_ptr()
    opts.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.fa_fwd(*args)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return out, lse, workspace


def fa_fwd_debug_dump(q, k, v, seq, head, row_tile, *, cu_seqlens_q=None, cu_seqlens_k=None, window_left=-1,
                      window_right=-1, softcap=0.0, scale=None, causal=False, max_seqlen_q=None,
                      max_seqlen_k=None, stream=None, **_):
    """fa_fwd through the prefill kernel's debug build, which also copies the
    intermediate values of the 128 query rows of tile ``row_tile`` of sequence
    ``seq``, q-head ``head``.  Returns ``(out, lse, workspace, dump)`` with
    ``dump = {"S": [n, 128, 128], "P": [n, 128, 128], "ref": [n, 128]}`` (fp32,
    entry it = the it-th key tile in the unit's list; n = the plan's n_k_tiles;
    entries past the list's end are unwritten)."""
    if not q.is_cuda:
        raise FaError(FA_ERR_INVALID_ARG, "fa_fwd_debug_dump (tensors must be CUDA tensors)")
    kw = dict(cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k, window_left=window_left,
              window_right=window_right, softcap=softcap, scale=scale, causal=causal, max_seqlen_q=max_seqlen_q,
              max_seqlen_k=max_seqlen_k)
    rc, plan = fa_fwd_plan(q, k, v, **kw)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_debug_dump (plan)")
    n_kt = plan["n_k_tiles"]
    dump = torch.empty(lib.fa_debug_dump_bytes(n_kt) // 4, dtype=torch.float32, device=q.device)
    oshape, lshape = _out_shapes(q, cu_seqlens_q, max_seqlen_q)
    out = torch.empty(oshape, dtype=q.dtype, device=q.device)
    lse = torch.empty(lshape, dtype=torch.float32, device=q.device)
    workspace = alloc_workspace(plan["workspace_bytes"], q.device)
    opts = make_opts(stream=stream, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k)
    opts.workspace = workspace.data_ptr()
    opts.workspace_bytes = workspace.numel() * workspace.element_size()
    descs = [describe(x) for x in (q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k)]
    rc = lib.fa_fwd_debug_dump(*[_ref(x) for x in descs], int(window_left), int(window_right), float(softcap),
                               float(scale or 0.0), int(bool(causal)), ctypes.byref(opts), int(seq), int(head),
                               int(row_tile), dump.data_ptr(), dump.numel() * 4)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_debug_dump")
    s_len = n_kt * 128 * 128
    parts = {"S": dump[:s_len].view(n_kt, 128, 128), "P": dump[s_len:2 * s_len].view(n_kt, 128, 128),
             "ref": dump[2 * s_len:2 * s_len + n_kt * 128].view(n_kt, 128)}
    return out, lse, workspace, parts


def fa_debug_dump_bytes_of(n_k_tiles: int) -> int:
    """Bytes fa_fwd_debug_dump needs for a plan with ``n_k_tiles`` key tiles."""
    return int(lib.fa_debug_dump_bytes(int(n_k_tiles)))


def _kv_args(q, k_cache, v_cache, k_new, v_new, out, lse, cu_seqlens_q, cache_seqlens, block_table,
             window_left, window_right, softcap, scale, causal, append, opts):
    descs = [describe(x) for x in (q, k_cache, v_cache, k_new, v_new, out, lse, cu_seqlens_q,
                                   cache_seqlens, block_table)]
    args = [_ref(x) for x in descs] + [int(window_left), int(window_right), float(softcap),
                                       float(scale or 0.0), int(bool(causal)), int(bool(append)),
                                       ctypes.byref(opts)]
    return args, (descs, opts)


def fa_fwd_kvcache_plan(q, k_cache, v_cache, k_new, v_new, cache_seqlens, *, out=None, lse=None,
                        cu_seqlens_q=None, block_table=None, window_left=-1, window_right=-1,
                        softcap=0.0, scale=None, causal=True, append=False, max_seqlen_q=None,
                        max_seqlen_k=None, debug_flags=0, stream=0, **_):
    """Host-only plan query of fa_fwd_kvcache; returns (status, plan dict)."""
    if out is None:
        out = q
    if lse is None:
        lse = torch.empty(_out_shapes(q, cu_seqlens_q, max_seqlen_q)[1], dtype=torch.float32,
                          device=q.device)
    opts = make_opts(stream=stream, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                     debug_flags=debug_flags)
    args, keep = _kv_args(q, k_cache, v_cache, k_new, v_new, out, lse, cu_seqlens_q, cache_seqlens,
                          block_table, window_left, window_right, softcap, scale, causal, append, opts)
    plan = fa_plan()
    rc = lib.fa_fwd_kvcache_plan(*args, ctypes.byref(plan))
    return rc, plan.as_dict()


def fa_fwd_kvcache(q, k_cache, v_cache, k_new, v_new, cache_seqlens, *, out=None, lse=None,
                   cu_seqlens_q=None, block_table=None, window_left=-1, window_right=-1, softcap=0.0,
                   scale=None, causal=True, append=False, max_seqlen_q=None, max_seqlen_k=None,
                   workspace=None, stream=None, debug_flags=0, event_begin=None, event_end=None,
                   alibi_slopes=None, event_attn_end=None, **_):
    """Attention over a KV cache plus the step's active keys (fa_fwd_kvcache of
    the C ABI): sequence s sees cache rows [0, cache_seqlens[s]) and then its
    own active rows ``k_new``/``v_new`` (laid out like ``q``); with ``append``
    the active rows are also written into the cache after the cached ones.
    ``max_seqlen_k`` (the largest cached + active count) is required.  Returns
    ``(out, lse, workspace)``; raises FaError on a non-zero status."""
    if not q.is_cuda:
        raise FaError(FA_ERR_INVALID_ARG, "fa_fwd_kvcache (tensors must be CUDA tensors)")
    oshape, lshape = _out_shapes(q, cu_seqlens_q, max_seqlen_q)
    if out is None:
        out = torch.empty(oshape, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(lshape, dtype=torch.float32, device=q.device)
    alibi_slopes = _alibi(alibi_slopes, q)
    opts = make_opts(stream=stream, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                     debug_flags=debug_flags, event_begin=event_begin, event_end=event_end,
                     alibi_slopes=alibi_slopes, event_attn_end=event_attn_end)
    args, keep = _kv_args(q, k_cache, v_cache, k_new, v_new, out, lse, cu_seqlens_q, cache_seqlens,
                          block_table, window_left, window_right, softcap, scale, causal, append, opts)
    if workspace is None:
        plan = fa_plan()
        rc = lib.fa_fwd_kvcache_plan(*args, ctypes.byref(plan))
        if rc != FA_OK:
            raise FaError(rc, "fa_fwd_kvcache_plan")
        workspace = alloc_workspace(plan.workspace_bytes, q.device)
    opts.workspace = workspace.data_ptr()
    opts.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.fa_fwd_kvcache(*args)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_kvcache")
    return out, lse, workspace


def _bwd_args(q, k, v, out, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, window_left, window_right,
              softcap, scale, causal, opts):
    descs = [describe(x) for x in (q, k, v, out, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k)]
    args = [_ref(x) for x in descs] + [int(window_left), int(window_right), float(softcap),
                                       float(scale or 0.0), int(bool(causal)), ctypes.byref(opts)]
    return args, (descs, opts)


def fa_bwd_plan(q, k, v, out, lse, dout, *, dq=None, dk=None, dv=None, cu_seqlens_q=None,
                cu_seqlens_k=None, window_left=-1, window_right=-1, softcap=0.0, scale=None,
                causal=False, max_seqlen_q=None, max_seqlen_k=None, debug_flags=0, stream=0, **_):
    """Host-only plan query of fa_bwd; returns (status, plan dict)."""
    dq = q if dq is None else dq
    dk = k if dk is None else dk
    dv = v if dv is None else dv
    opts = make_opts(stream=stream, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                     debug_flags=debug_flags)
    args, keep = _bwd_args(q, k, v, out, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, window_left,
                           window_right, softcap, scale, causal, opts)
    plan = fa_plan()
    rc = lib.fa_bwd_plan(*args, ctypes.byref(plan))
    return rc, plan.as_dict()


def fa_bwd(q, k, v, out, lse, dout, *, dq=None, dk=None, dv=None, cu_seqlens_q=None, cu_seqlens_k=None,
           window_left=-1, window_right=-1, softcap=0.0, scale=None, causal=False, max_seqlen_q=None,
           max_seqlen_k=None, workspace=None, stream=None, debug_flags=0, event_begin=None, event_end=None,
           alibi_slopes=None, **_):
    """Backward pass (fa_bwd of the C ABI): gradients of the forward for the
    same arguments, ``out`` and ``lse`` from fa_fwd and ``dout`` = dL/dout.
    Returns ``(dq, dk, dv, workspace)``; dq/dk/dv are allocated with torch when
    not given.  Raises FaError on a non-zero status."""
    if not q.is_cuda:
        raise FaError(FA_ERR_INVALID_ARG, "fa_bwd (tensors must be CUDA tensors)")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    alibi_slopes = _alibi(alibi_slopes, q)
    opts = make_opts(stream=stream, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                     debug_flags=debug_flags, event_begin=event_begin, event_end=event_end,
                     alibi_slopes=alibi_slopes)
    args, keep = _bwd_args(q, k, v, out, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, window_left,
                           window_right, softcap, scale, causal, opts)
    if workspace is None:
        plan = fa_plan()
        rc = lib.fa_bwd_plan(*args, ctypes.byref(plan))
        if rc != FA_OK:
            raise FaError(rc, "fa_bwd_plan")
        workspace = alloc_workspace(plan.workspace_bytes, q.device)
    opts.workspace = workspace.data_ptr()
    opts.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.fa_bwd(*args)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv, workspace


def fa_check_device_error(workspace, stream=None):
    """Synchronise and read/clear the device error word; returns (status, info)."""
    info = ctypes.c_uint32(0)
    st = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = lib.fa_check_device_error(st, workspace.data_ptr(), ctypes.byref(info))
    return rc, info.value


def fa_fwd_noalloc(q, k, v, *, out, lse, cu_seqlens_q=None, cu_seqlens_k=None, block_table=None,
                   mask=None, zero_hold_states=None, keep_window=0, window_left=-1, window_right=-1,
                   softcap=0.0, scale=None, causal=False, max_seqlen_q=None, max_seqlen_k=None,
                   stream=None, debug_flags=0, alibi_slopes=None, workspace=None, event_begin=None,
                   event_end=None, event_attn_end=None):
    """fa_fwd_noalloc of the C ABI: the forward pass for callers that may not
    allocate device memory.  ``out`` and ``lse`` are caller-provided; the
    library's static device scratch replaces the workspace, so nothing is
    allocated by this call.  A workspace or timing events cannot be used here
    and are refused rather than ignored.  Raises FaError on a non-zero status
    (a problem too large for the static scratch gives FA_ERR_WORKSPACE)."""
    if workspace is not None or event_begin is not None or event_end is not None or event_attn_end is not None:
        raise FaError(FA_ERR_INVALID_ARG, "fa_fwd_noalloc (takes no workspace and no timing events)")
    fn = lib.fa_fwd_noalloc
    alibi_slopes = _alibi(alibi_slopes, q)
    opts = make_opts(stream=stream, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                     debug_flags=debug_flags, alibi_slopes=alibi_slopes)
    args, keep = _args(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask,
                       zero_hold_states, keep_window, window_left, window_right, softcap,
                       scale or 0.0, causal, opts)
    rc = fn(*args)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_noalloc")
    return out, lse
