"""ctypes binding of ``include/ssd.h``: argument marshalling only.

Every numeric step runs in ``libssd_gb300.so``; torch supplies device memory
and the current stream.  The library is loaded on first use and a missing
build raises immediately -- there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssd_gb300.so")

SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_WORKSPACE, SSD_ERR_CUDA = range(5)
SSD_F32, SSD_BF16 = 0, 1
DEVERR_SLOT, DEVERR_METADATA, DEVERR_COLUMN, DEVERR_TIMEOUT, DEVERR_INTERNAL = 1, 2, 4, 8, 16

EXPORTED_SYMBOLS = ("ssd_status_string", "ssd_abi_version", "ssd_max_chunks", "ssd_chunk_metadata",
                    "ssd_prefill_workspace_size", "ssd_prefill_kernel_count", "ssd_prefill_varlen",
                    "ssd_prefill_varlen_marked", "ssd_prefill_varlen_noalloc", "ssm_decode_update", "ssd_mixed_step",
                    "ssd_conv1d_varlen",
                    "ssd_conv1d_update",
                    "mamba1_scan_varlen", "mamba1_state_update")

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_f32 = ctypes.c_float


class PrefillArgs(ctypes.Structure):
    _fields_ = [("total_tokens", _i32), ("num_seqs", _i32), ("num_chunks", _i32), ("nheads", _i32),
                ("headdim", _i32), ("dstate", _i32), ("ngroups", _i32), ("chunk_size", _i32),
                ("dtype", _i32), ("dt_softplus", _i32), ("dt_min", _f32), ("dt_max", _f32),
                ("num_slots", _i32), ("null_block_id", _i32),
                ("x", _vp), ("dt", _vp), ("B", _vp), ("C", _vp), ("z", _vp), ("A", _vp), ("D", _vp),
                ("dt_bias", _vp), ("cu_seqlens", _vp), ("cu_chunk_seqlens", _vp), ("seq_idx", _vp),
                ("last_chunk_indices", _vp), ("init_slot", _vp), ("chunk_slot", _vp),
                ("state_cache", _vp), ("y", _vp), ("err_word", _vp), ("seq_order", _vp),
                ("wait_limit_cycles", ctypes.c_int64)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("batch", _i32), ("tokens_per_req", _i32), ("nheads", _i32), ("headdim", _i32),
                ("dstate", _i32), ("ngroups", _i32), ("dtype", _i32), ("dt_softplus", _i32),
                ("dt_min", _f32), ("dt_max", _f32), ("num_slots", _i32), ("null_block_id", _i32),
                ("state_indices_cols", _i32),
                ("x", _vp), ("dt", _vp), ("B", _vp), ("C", _vp), ("z", _vp), ("A", _vp), ("D", _vp),
                ("dt_bias", _vp), ("state_cache", _vp), ("state_indices", _vp),
                ("num_accepted_tokens", _vp), ("y", _vp), ("err_word", _vp)]


class Conv1dArgs(ctypes.Structure):
    _fields_ = [("total_tokens", _i32), ("num_seqs", _i32), ("num_chunks", _i32), ("tokens_per_req", _i32),
                ("dim_x", _i32), ("dim_bc", _i32), ("width", _i32), ("dtype", _i32), ("activation", _i32),
                ("num_slots", _i32), ("null_block_id", _i32),
                ("xbc", _vp), ("weight", _vp), ("bias", _vp), ("cu_seqlens", _vp), ("cu_chunk_seqlens", _vp),
                ("last_chunk_indices", _vp), ("init_slot", _vp), ("out_slot", _vp), ("chunk_slot", _vp),
                ("conv_state", _vp), ("x_out", _vp), ("B_out", _vp), ("C_out", _vp), ("err_word", _vp)]


class Mamba1Args(ctypes.Structure):
    _fields_ = [("total_tokens", _i32), ("num_seqs", _i32), ("num_chunks", _i32), ("tokens_per_req", _i32),
                ("dim", _i32), ("dstate", _i32), ("ngroups", _i32), ("dtype", _i32), ("dt_softplus", _i32),
                ("dt_min", _f32), ("dt_max", _f32), ("num_slots", _i32), ("null_block_id", _i32),
                ("state_indices_cols", _i32),
                ("x", _vp), ("dt", _vp), ("B", _vp), ("C", _vp), ("z", _vp), ("A", _vp), ("D", _vp),
                ("dt_bias", _vp), ("cu_seqlens", _vp), ("cu_chunk_seqlens", _vp), ("last_chunk_indices", _vp),
                ("init_slot", _vp), ("chunk_slot", _vp), ("state_indices", _vp), ("num_accepted_tokens", _vp),
                ("state_cache", _vp), ("y", _vp), ("err_word", _vp)]


class SSDError(RuntimeError):
    def __init__(self, fn, code):
        name = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED",
                3: "SSD_ERR_WORKSPACE", 4: "SSD_ERR_CUDA"}.get(code, str(code))
        super().__init__("%s returned %s" % (fn, name))
        self.code = code


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("%s is missing: build it with __graft_entry__.build() (nvcc, sm_103a)"
                               % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        ip = ctypes.POINTER(ctypes.c_int32)
        L.ssd_status_string.restype = ctypes.c_char_p
        L.ssd_status_string.argtypes = [ctypes.c_int]
        L.ssd_abi_version.restype = _i32
        L.ssd_max_chunks.restype = _i32
        L.ssd_max_chunks.argtypes = [_i32, _i32, _i32]
        L.ssd_chunk_metadata.restype = ctypes.c_int
        L.ssd_chunk_metadata.argtypes = [_i32, _i32, ip, ip, ctypes.POINTER(ctypes.c_uint8), ip,
                                         ctypes.c_int64, _i32, ip, _i32, _i32, ip, ip, ip, ip, ip,
                                         ip, ip, ip]
        L.ssd_prefill_workspace_size.restype = ctypes.c_size_t
        L.ssd_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
        L.ssd_prefill_kernel_count.restype = _i32
        L.ssd_prefill_kernel_count.argtypes = [ctypes.POINTER(PrefillArgs)]
        L.ssd_prefill_varlen.restype = ctypes.c_int
        L.ssd_prefill_varlen.argtypes = [ctypes.POINTER(PrefillArgs), _vp, ctypes.c_size_t, _vp]
        L.ssd_prefill_varlen_marked.restype = ctypes.c_int
        L.ssd_prefill_varlen_marked.argtypes = [ctypes.POINTER(PrefillArgs), _vp, ctypes.c_size_t, _vp, _vp]
        L.ssd_prefill_varlen_noalloc.restype = ctypes.c_int
        L.ssd_prefill_varlen_noalloc.argtypes = [ctypes.POINTER(PrefillArgs), _vp]
        L.ssm_decode_update.restype = ctypes.c_int
        L.ssm_decode_update.argtypes = [ctypes.POINTER(DecodeArgs), _vp]
        L.ssd_mixed_step.restype = ctypes.c_int
        L.ssd_mixed_step.argtypes = [ctypes.POINTER(PrefillArgs), _vp, ctypes.c_size_t,
                                     ctypes.POINTER(DecodeArgs), _vp]
        for fn in ("mamba1_scan_varlen", "mamba1_state_update"):
            getattr(L, fn).restype = ctypes.c_int
            getattr(L, fn).argtypes = [ctypes.POINTER(Mamba1Args), _vp]
        _lib = L
    return _lib


# ----------------------------------------------------------------- helpers --

def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    if t.dtype == torch.float32:
        return SSD_F32
    raise ValueError("x/dt/B/C must be bfloat16 or float32, got %s" % t.dtype)


def _dev(t, name, dtype=None, required=True):
    if t is None:
        if required:
            raise ValueError("%s is required" % name)
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _host_i32(a, name):
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        if a.is_cuda:
            raise ValueError("%s must be host memory" % name)
        a = a.numpy()
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _ptr(a, ctype=ctypes.c_int32):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ----------------------------------------------------------------- API ------

def ssd_max_chunks(num_seqs, total_tokens, chunk_size):
    return int(lib().ssd_max_chunks(int(num_seqs), int(total_tokens), int(chunk_size)))


def ssd_chunk_metadata(cu_seqlens, chunk_size, num_computed_tokens=None, has_initial_states=None,
                       block_table=None, state_indices=None, null_block_id=0):
    """Host chunk metadata and slot routing (see ``ssd_chunk_metadata`` in ssd.h).

    All inputs are host arrays; returns a dict of int32 numpy arrays:
    cu_chunk_seqlens [K+1], seq_idx [K], last_chunk_indices [S],
    chunk_block_col [K], init_slot [S], chunk_slot [K], seq_order [S].
    """
    cu = _host_i32(cu_seqlens, "cu_seqlens")
    S = cu.shape[0] - 1
    T = int(cu[-1])
    nc = _host_i32(num_computed_tokens, "num_computed_tokens")
    has = None
    if has_initial_states is not None:
        h = has_initial_states.numpy() if isinstance(has_initial_states, torch.Tensor) else has_initial_states
        has = np.ascontiguousarray(np.asarray(h).astype(bool), dtype=np.uint8)
    bt = _host_i32(block_table, "block_table")
    si = _host_i32(state_indices, "state_indices")
    maxk = max(ssd_max_chunks(S, T, chunk_size), 0)
    out = dict(cu_chunk_seqlens=np.zeros(maxk + 1, np.int32), seq_idx=np.zeros(max(maxk, 1), np.int32),
               last_chunk_indices=np.zeros(max(S, 1), np.int32),
               chunk_block_col=np.zeros(max(maxk, 1), np.int32), init_slot=np.zeros(max(S, 1), np.int32),
               chunk_slot=np.zeros(max(maxk, 1), np.int32), seq_order=np.zeros(max(S, 1), np.int32))
    k = ctypes.c_int32(0)
    rc = lib().ssd_chunk_metadata(
        S, int(chunk_size), _ptr(cu), _ptr(nc), _ptr(has, ctypes.c_uint8), _ptr(bt),
        0 if bt is None else bt.shape[1], 0 if bt is None else bt.shape[1], _ptr(si), int(null_block_id),
        maxk, _ptr(out["cu_chunk_seqlens"]), _ptr(out["seq_idx"]), _ptr(out["last_chunk_indices"]),
        _ptr(out["chunk_block_col"]), _ptr(out["init_slot"]), _ptr(out["chunk_slot"]), _ptr(out["seq_order"]),
        ctypes.byref(k))
    if rc != SSD_OK:
        raise SSDError("ssd_chunk_metadata", rc)
    K = k.value
    return dict(cu_chunk_seqlens=out["cu_chunk_seqlens"][:K + 1].copy(), seq_idx=out["seq_idx"][:K].copy(),
                last_chunk_indices=out["last_chunk_indices"][:S].copy(),
                chunk_block_col=out["chunk_block_col"][:K].copy(), init_slot=out["init_slot"][:S].copy(),
                chunk_slot=out["chunk_slot"][:K].copy(), seq_order=out["seq_order"][:S].copy())


def prefill_args(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, seq_idx, last_chunk_indices, out,
                 init_slot=None, chunk_slot=None, state_cache=None, D=None, dt_bias=None, z=None,
                 dt_softplus=True, dt_limit=(0.0, math.inf), null_block_id=0, chunk_size=None,
                 err_word=None, seq_order=None, wait_limit_cycles=0):
    """Fills a ``PrefillArgs`` from device tensors (validating shapes and dtypes)."""
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    dtype = _dtype_code(x)
    for name, t, shp in (("dt", dt, (T, H)), ("B", B, (T, G, N)), ("C", C, (T, G, N)), ("out", out, (T, H, P))):
        if tuple(t.shape) != shp or t.dtype != x.dtype:
            raise ValueError("%s must be %s of shape %s" % (name, x.dtype, shp))
    S = cu_seqlens.shape[0] - 1
    K = cu_chunk_seqlens.shape[0] - 1
    a = PrefillArgs()
    a.total_tokens, a.num_seqs, a.num_chunks = T, S, K
    a.nheads, a.headdim, a.dstate, a.ngroups = H, P, N, G
    a.chunk_size = int(chunk_size) if chunk_size else 0
    a.dtype = dtype
    a.dt_softplus = int(bool(dt_softplus))
    a.dt_min, a.dt_max = float(dt_limit[0]), float(dt_limit[1])
    a.null_block_id = int(null_block_id)
    a.x, a.dt, a.B, a.C, a.y = (_dev(x, "x"), _dev(dt, "dt"), _dev(B, "B"), _dev(C, "C"), _dev(out, "out"))
    a.z = _dev(z, "z", required=False)
    a.A = _dev(A, "A", torch.float32)
    a.D = _dev(D, "D", torch.float32, required=False)
    a.dt_bias = _dev(dt_bias, "dt_bias", torch.float32, required=False)
    a.cu_seqlens = _dev(cu_seqlens, "cu_seqlens", torch.int32)
    a.cu_chunk_seqlens = _dev(cu_chunk_seqlens, "cu_chunk_seqlens", torch.int32)
    a.seq_idx = _dev(seq_idx, "seq_idx", torch.int32, required=False)
    a.last_chunk_indices = _dev(last_chunk_indices, "last_chunk_indices", torch.int32)
    a.init_slot = _dev(init_slot, "init_slot", torch.int32, required=False)
    a.chunk_slot = _dev(chunk_slot, "chunk_slot", torch.int32, required=False)
    if state_cache is not None:
        if state_cache.dtype != torch.float32 or tuple(state_cache.shape[1:]) != (H, P, N):
            raise ValueError("state_cache must be float32 [slots, %d, %d, %d]" % (H, P, N))
        a.state_cache = _dev(state_cache, "state_cache")
        a.num_slots = state_cache.shape[0]
    a.err_word = _dev(err_word, "err_word", required=False)
    a.seq_order = _dev(seq_order, "seq_order", torch.int32, required=False)
    a.wait_limit_cycles = int(wait_limit_cycles)
    if a.chunk_size == 0:
        a.chunk_size = 1
    return a


def ssd_prefill_workspace_size(args):
    return int(lib().ssd_prefill_workspace_size(ctypes.byref(args)))


def ssd_prefill_kernel_count(args):
    return int(lib().ssd_prefill_kernel_count(ctypes.byref(args)))


def ssd_prefill_varlen(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, seq_idx, last_chunk_indices,
                       out=None, init_slot=None, chunk_slot=None, state_cache=None, D=None,
                       dt_bias=None, z=None, dt_softplus=True, dt_limit=(0.0, math.inf),
                       null_block_id=0, chunk_size=None, workspace=None, err_word=None, stream=None,
                       seq_order=None, wait_limit_cycles=0, mark=None):
    """Varlen SSD prefill on device tensors; returns ``out`` ([T,H,P], x's dtype).

    ``workspace`` (uint8 CUDA tensor) is allocated with torch when omitted.  ``mark``: a
    ``torch.cuda.Event`` the library records right before the call's main kernel
    (``ssd_prefill_varlen_marked``), for timing the call's kernels apart.
    """
    if out is None:
        out = torch.empty_like(x)
    a = prefill_args(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, seq_idx, last_chunk_indices, out,
                     init_slot, chunk_slot, state_cache, D, dt_bias, z, dt_softplus, dt_limit,
                     null_block_id, chunk_size, err_word, seq_order, wait_limit_cycles)
    need = ssd_prefill_workspace_size(a)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    if mark is None:
        rc = lib().ssd_prefill_varlen(ctypes.byref(a), ctypes.c_void_p(workspace.data_ptr()),
                                      workspace.numel(), _stream(stream))
    else:
        if not mark.cuda_event:  # torch makes its events on their first record
            mark.record()
        rc = lib().ssd_prefill_varlen_marked(ctypes.byref(a), ctypes.c_void_p(workspace.data_ptr()),
                                             workspace.numel(), _stream(stream), ctypes.c_void_p(mark.cuda_event))
    if rc != SSD_OK:
        raise SSDError("ssd_prefill_varlen", rc)
    return out


def decode_args(x, dt, A, B, C, state_cache, state_indices, out, num_accepted_tokens=None, D=None,
                dt_bias=None, z=None, dt_softplus=True, dt_limit=(0.0, math.inf), null_block_id=0,
                err_word=None):
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    R, cols = state_indices.shape
    if R == 0 or T % R:
        raise ValueError("x rows must be a multiple of state_indices rows")
    for name, t, shp in (("dt", dt, (T, H)), ("B", B, (T, G, N)), ("C", C, (T, G, N)), ("out", out, (T, H, P))):
        if tuple(t.shape) != shp or t.dtype != x.dtype:
            raise ValueError("%s must be %s of shape %s" % (name, x.dtype, shp))
    if state_cache.dtype != torch.float32 or tuple(state_cache.shape[1:]) != (H, P, N):
        raise ValueError("state_cache must be float32 [slots, %d, %d, %d]" % (H, P, N))
    a = DecodeArgs()
    a.batch, a.tokens_per_req = R, T // R
    a.nheads, a.headdim, a.dstate, a.ngroups = H, P, N, G
    a.dtype = _dtype_code(x)
    a.dt_softplus = int(bool(dt_softplus))
    a.dt_min, a.dt_max = float(dt_limit[0]), float(dt_limit[1])
    a.num_slots = state_cache.shape[0]
    a.null_block_id = int(null_block_id)
    a.state_indices_cols = cols
    a.x, a.dt, a.B, a.C, a.y = (_dev(x, "x"), _dev(dt, "dt"), _dev(B, "B"), _dev(C, "C"), _dev(out, "out"))
    a.z = _dev(z, "z", required=False)
    a.A = _dev(A, "A", torch.float32)
    a.D = _dev(D, "D", torch.float32, required=False)
    a.dt_bias = _dev(dt_bias, "dt_bias", torch.float32, required=False)
    a.state_cache = _dev(state_cache, "state_cache")
    a.state_indices = _dev(state_indices, "state_indices", torch.int32)
    a.num_accepted_tokens = _dev(num_accepted_tokens, "num_accepted_tokens", torch.int32, required=False)
    a.err_word = _dev(err_word, "err_word", required=False)
    return a


def ssm_decode_update(x, dt, A, B, C, state_cache, state_indices, num_accepted_tokens=None, out=None,
                      D=None, dt_bias=None, z=None, dt_softplus=True, dt_limit=(0.0, math.inf),
                      null_block_id=0, err_word=None, stream=None):
    """In-place decode update of ``state_cache``; returns ``out`` ([R*tpr,H,P])."""
    if out is None:
        out = torch.empty_like(x)
    a = decode_args(x, dt, A, B, C, state_cache, state_indices, out, num_accepted_tokens, D, dt_bias, z,
                    dt_softplus, dt_limit, null_block_id, err_word)
    rc = lib().ssm_decode_update(ctypes.byref(a), _stream(stream))
    if rc != SSD_OK:
        raise SSDError("ssm_decode_update", rc)
    return out


def ssd_mixed_step(prefill, decode, workspace=None, stream=None):
    """One step of a mixed batch: ``prefill`` (from :func:`prefill_args`) and ``decode`` (from
    :func:`decode_args`) issued together on ``stream``; the tensors the two argument sets point
    to must stay alive until the step is done.  ``workspace`` as for :func:`ssd_prefill_varlen`
    (allocated with torch when omitted)."""
    if workspace is None:
        need = ssd_prefill_workspace_size(prefill) if prefill.total_tokens > 0 else 0
        dev = torch.device("cuda", torch.cuda.current_device())
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    rc = lib().ssd_mixed_step(ctypes.byref(prefill), ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                              ctypes.byref(decode), _stream(stream))
    if rc != SSD_OK:
        raise SSDError("ssd_mixed_step", rc)


def conv1d_args(xbc, weight, dim_x, dim_bc, x_out, B_out, C_out, bias=None, conv_state=None, activation="silu",
                null_block_id=0, err_word=None):
    """Arguments shared by the two conv calls (sizes, tensors, activation)."""
    T, D = xbc.shape
    if D != dim_x + 2 * dim_bc:
        raise ValueError("xbc has %d channels, dim_x + 2 dim_bc = %d" % (D, dim_x + 2 * dim_bc))
    if weight.dtype != torch.float32 or weight.dim() != 2 or weight.shape[0] != D:
        raise ValueError("weight must be float32 [%d, W]" % D)
    W = weight.shape[1]
    for name, t, shp in (("x_out", x_out, (T, dim_x)), ("B_out", B_out, (T, dim_bc)), ("C_out", C_out, (T, dim_bc))):
        if tuple(t.shape) != shp or t.dtype != xbc.dtype:
            raise ValueError("%s must be %s of shape %s" % (name, xbc.dtype, shp))
    if conv_state is not None and (conv_state.dtype != xbc.dtype or tuple(conv_state.shape[1:]) != (W - 1, D)):
        raise ValueError("conv_state must be %s [slots, %d, %d]" % (xbc.dtype, W - 1, D))
    a = Conv1dArgs()
    a.total_tokens, a.dim_x, a.dim_bc, a.width = T, dim_x, dim_bc, W
    a.dtype = _dtype_code(xbc)
    a.activation = {"silu": 1, None: 0, "none": 0}[activation]
    a.num_slots = 0 if conv_state is None else conv_state.shape[0]
    a.null_block_id = int(null_block_id)
    a.xbc = _dev(xbc, "xbc")
    a.weight = _dev(weight, "weight", torch.float32)
    a.bias = _dev(bias, "bias", torch.float32, required=False)
    a.conv_state = _dev(conv_state, "conv_state", required=False)
    a.x_out, a.B_out, a.C_out = _dev(x_out, "x_out"), _dev(B_out, "B_out"), _dev(C_out, "C_out")
    a.err_word = _dev(err_word, "err_word", required=False)
    return a


def _conv_outputs(xbc, dim_x, dim_bc, x_out, B_out, C_out):
    T = xbc.shape[0]
    if x_out is None:
        x_out = torch.empty((T, dim_x), dtype=xbc.dtype, device=xbc.device)
    if B_out is None:
        B_out = torch.empty((T, dim_bc), dtype=xbc.dtype, device=xbc.device)
    if C_out is None:
        C_out = torch.empty((T, dim_bc), dtype=xbc.dtype, device=xbc.device)
    return x_out, B_out, C_out


def ssd_conv1d_varlen(xbc, weight, cu_seqlens, dim_x, dim_bc, bias=None, conv_state=None, init_slot=None,
                      out_slot=None, chunk_slot=None, cu_chunk_seqlens=None, last_chunk_indices=None,
                      activation="silu", null_block_id=0, x_out=None, B_out=None, C_out=None, err_word=None,
                      stream=None):
    """Depthwise causal conv1d over packed sequences; returns (x [T, dim_x], B [T, dim_bc],
    C [T, dim_bc]).  Device int32 metadata as for ssd_prefill_varlen."""
    x_out, B_out, C_out = _conv_outputs(xbc, dim_x, dim_bc, x_out, B_out, C_out)
    a = conv1d_args(xbc, weight, dim_x, dim_bc, x_out, B_out, C_out, bias, conv_state, activation,
                    null_block_id, err_word)
    a.num_seqs = cu_seqlens.numel() - 1
    a.num_chunks = 0 if cu_chunk_seqlens is None else cu_chunk_seqlens.numel() - 1
    a.cu_seqlens = _dev(cu_seqlens, "cu_seqlens", torch.int32)
    a.cu_chunk_seqlens = _dev(cu_chunk_seqlens, "cu_chunk_seqlens", torch.int32, required=False)
    a.last_chunk_indices = _dev(last_chunk_indices, "last_chunk_indices", torch.int32, required=False)
    a.init_slot = _dev(init_slot, "init_slot", torch.int32, required=False)
    a.out_slot = _dev(out_slot, "out_slot", torch.int32, required=False)
    a.chunk_slot = _dev(chunk_slot, "chunk_slot", torch.int32, required=False)
    rc = lib().ssd_conv1d_varlen(ctypes.byref(a), _stream(stream))
    if rc != SSD_OK:
        raise SSDError("ssd_conv1d_varlen", rc)
    return x_out, B_out, C_out


def ssd_conv1d_update(xbc, weight, conv_state, state_indices, dim_x, dim_bc, bias=None, activation="silu",
                      null_block_id=0, x_out=None, B_out=None, C_out=None, err_word=None, stream=None):
    """Decode conv step: request r's rows r*tpr .. r*tpr + tpr - 1 continue the conv state in slot
    state_indices[r], which then holds the state after its last token; null rows are padding."""
    R = state_indices.numel()
    T = xbc.shape[0]
    if R == 0 or T % R:
        raise ValueError("xbc rows must be a multiple of the requests")
    x_out, B_out, C_out = _conv_outputs(xbc, dim_x, dim_bc, x_out, B_out, C_out)
    a = conv1d_args(xbc, weight, dim_x, dim_bc, x_out, B_out, C_out, bias, conv_state, activation,
                    null_block_id, err_word)
    a.num_seqs, a.tokens_per_req = R, T // R
    a.init_slot = _dev(state_indices, "state_indices", torch.int32)
    rc = lib().ssd_conv1d_update(ctypes.byref(a), _stream(stream))
    if rc != SSD_OK:
        raise SSDError("ssd_conv1d_update", rc)
    return x_out, B_out, C_out


# ------------------------------------------------------------------ Mamba1 --

def mamba1_args(x, dt, A, B, C, y, D=None, dt_bias=None, z=None, state_cache=None, dt_softplus=True,
                dt_limit=(0.0, math.inf), null_block_id=0, err_word=None):
    """Arguments shared by the two Mamba1 calls: x, dt, z, y [T, Dc]; B, C [T, G, N]; A [Dc, N]
    float32; D, dt_bias [Dc] float32; state_cache [slots, Dc, N] float32."""
    T, Dc = x.shape
    if B.dim() != 3 or B.shape[0] != T:
        raise ValueError("B must be [T, G, N]")
    G, N = B.shape[1], B.shape[2]
    for name, t, shp in (("dt", dt, (T, Dc)), ("C", C, (T, G, N)), ("y", y, (T, Dc))) + \
            ((("z", z, (T, Dc)),) if z is not None else ()):
        if tuple(t.shape) != shp or t.dtype != x.dtype:
            raise ValueError("%s must be %s of shape %s" % (name, x.dtype, shp))
    if tuple(A.shape) != (Dc, N):
        raise ValueError("A must be [%d, %d]" % (Dc, N))
    if state_cache is not None and tuple(state_cache.shape[1:]) != (Dc, N):
        raise ValueError("state_cache must be [slots, %d, %d]" % (Dc, N))
    a = Mamba1Args()
    a.total_tokens, a.dim, a.dstate, a.ngroups = T, Dc, N, G
    a.dtype = _dtype_code(x)
    a.dt_softplus = int(bool(dt_softplus))
    a.dt_min, a.dt_max = float(dt_limit[0]), float(dt_limit[1])
    a.num_slots = 0 if state_cache is None else state_cache.shape[0]
    a.null_block_id = int(null_block_id)
    a.x, a.dt, a.B, a.C, a.y = _dev(x, "x"), _dev(dt, "dt"), _dev(B, "B"), _dev(C, "C"), _dev(y, "y")
    a.z = _dev(z, "z", required=False)
    a.A = _dev(A, "A", torch.float32)
    a.D = _dev(D, "D", torch.float32, required=False)
    a.dt_bias = _dev(dt_bias, "dt_bias", torch.float32, required=False)
    a.state_cache = _dev(state_cache, "state_cache", torch.float32, required=False)
    a.err_word = _dev(err_word, "err_word", required=False)
    return a


def mamba1_scan_varlen(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, last_chunk_indices, D=None, dt_bias=None,
                       z=None, state_cache=None, init_slot=None, chunk_slot=None, dt_softplus=True,
                       dt_limit=(0.0, math.inf), null_block_id=0, out=None, err_word=None, stream=None):
    """Mamba1 selective scan over packed sequences; returns y [T, Dc].  Device int32 metadata
    from ssd_chunk_metadata (chunk_size 2048 is Mamba1's default); state_cache updated in place."""
    if out is None:
        out = torch.empty_like(x)
    a = mamba1_args(x, dt, A, B, C, out, D, dt_bias, z, state_cache, dt_softplus, dt_limit, null_block_id,
                    err_word)
    a.num_seqs = cu_seqlens.numel() - 1
    a.num_chunks = cu_chunk_seqlens.numel() - 1
    a.cu_seqlens = _dev(cu_seqlens, "cu_seqlens", torch.int32)
    a.cu_chunk_seqlens = _dev(cu_chunk_seqlens, "cu_chunk_seqlens", torch.int32)
    a.last_chunk_indices = _dev(last_chunk_indices, "last_chunk_indices", torch.int32)
    a.init_slot = _dev(init_slot, "init_slot", torch.int32, required=False)
    a.chunk_slot = _dev(chunk_slot, "chunk_slot", torch.int32, required=False)
    rc = lib().mamba1_scan_varlen(ctypes.byref(a), _stream(stream))
    if rc != SSD_OK:
        raise SSDError("mamba1_scan_varlen", rc)
    return out


def mamba1_state_update(x, dt, A, B, C, state_cache, state_indices, num_accepted_tokens=None, out=None, D=None,
                        dt_bias=None, z=None, dt_softplus=True, dt_limit=(0.0, math.inf), null_block_id=0,
                        err_word=None, stream=None):
    """Mamba1 decode: in-place update of ``state_cache`` through ``state_indices`` [R, cols];
    returns y [R * tpr, Dc]."""
    if out is None:
        out = torch.empty_like(x)
    if state_indices.dim() != 2:
        raise ValueError("state_indices must be [R, cols]")
    R, cols = state_indices.shape
    T = x.shape[0]
    if R == 0 or T % R:
        raise ValueError("x rows must be a multiple of the requests")
    a = mamba1_args(x, dt, A, B, C, out, D, dt_bias, z, state_cache, dt_softplus, dt_limit, null_block_id,
                    err_word)
    a.num_seqs, a.tokens_per_req, a.state_indices_cols = R, T // R, cols
    a.state_indices = _dev(state_indices, "state_indices", torch.int32)
    a.num_accepted_tokens = _dev(num_accepted_tokens, "num_accepted_tokens", torch.int32, required=False)
    rc = lib().mamba1_state_update(ctypes.byref(a), _stream(stream))
    if rc != SSD_OK:
        raise SSDError("mamba1_state_update", rc)
    return out
