"""CPU oracle for the selective-SSM prefill and decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may
import this package.  The CUDA library never imports, links or calls it, and
the two share no code: this package holds a plain C implementation
(``ssd_oracle.c``, fp64, strictly sequential in time) plus the index routing
written as plain Python loops.

Sources it follows (page titles and sections):

* [vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링 -- "논문 핵심 내용"
  (selective SSM: Delta, B, C depend on the input), "청크 메타데이터 계산"
  (chunks hold one sequence; the state is taken every chunk_size tokens),
  "CUDA Graph 지원" (padded decode rows carry NULL_BLOCK_ID),
  "왜 이 설계인가" items 2 and 4 (decode is a sequential update; spec-decode
  resumes from the checkpoint chosen by num_accepted_tokens),
  "MetadataBuilder 초기화" (decode state-index table of 1 + num_spec columns,
  or one column per block in "all" cache mode).
* [vllm] vLLM Mamba2 SSD 커널 웜업 -- "mamba_mixer2.py 변경 사항 (핵심)"
  (the varlen chunk-scan call: shapes, dt_bias, dt_softplus, dt_limit, D,
  initial states in the state dtype).

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, invariants and independent evaluations; see the docstrings.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libssd_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``ssd_oracle.c`` with gcc into ``oracle/_build``."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp,
                               _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        up = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_ssd_prefill.restype = ctypes.c_int
        lib.oracle_ssd_prefill.argtypes = [
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int32, ctypes.c_double,
            ctypes.c_double, ip, ctypes.c_int32, ip, dp, up, dp, dp, dp, ctypes.c_int32]
        lib.oracle_mamba1_prefill.restype = ctypes.c_int
        lib.oracle_mamba1_prefill.argtypes = [
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            dp, dp, dp, dp, dp, dp, dp, ctypes.c_int32, ctypes.c_double, ctypes.c_double,
            ip, ctypes.c_int32, ip, dp, up, dp, dp, dp, ctypes.c_int32]
        lib.oracle_chunk_metadata.restype = ctypes.c_int32
        lib.oracle_chunk_metadata.argtypes = [ctypes.c_int32, ctypes.c_int32, ip, ip,
                                              ctypes.c_int32, ip, ip, ip, ip]
        lib.oracle_delta_value.restype = ctypes.c_double
        lib.oracle_delta_value.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_double]
        _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def delta(dt, bias, dt_softplus=True, dt_limit=(0.0, math.inf)):
    """Scalar Delta = clamp(softplus(dt + bias), *dt_limit) as the C oracle forms it."""
    return _load().oracle_delta_value(float(dt), float(bias), int(bool(dt_softplus)),
                                      float(dt_limit[0]), float(dt_limit[1]))


def silu(z):
    """silu(z) = z * sigmoid(z), in fp64, with sigmoid(z) = 1 / (1 + e) for
    z >= 0 and e / (1 + e) for z < 0, e = exp(-|z|): neither branch
    overflows, and neither subtracts nearly equal numbers.

    The output gate: the chunk-scan call of "[vllm] vLLM Mamba2 SSD 커널 웜업"
    ("mamba_mixer2.py 변경 사항 (핵심)") takes an optional z (None in the
    warm-up); as in Mamba2, a gated output is y * silu(z) elementwise.
    """
    z = _f64(z)
    e = np.exp(-np.abs(z))
    return z * np.where(z >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def ssd_prefill(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens=None, D=None, dt_bias=None,
                initial_states=None, has_initial_states=None, dt_softplus=True,
                dt_limit=(0.0, math.inf), nthreads=None, z=None):
    """Sequential fp64 recurrence over packed varlen sequences.

    x [T,H,P], dt [T,H], B and C [T,G,N], A/D/dt_bias [H], cu_seqlens [S+1],
    cu_chunk_seqlens [K+1] (optional), initial_states [S,H,P,N] with the
    boolean has_initial_states [S].  Returns ``(y [T,H,P], chunk_states
    [K,H,P,N] or None, final_states [S,H,P,N])``, all fp64.  chunk_states[k]
    is the state right after the last token of chunk k.  With a gate z
    [T,H,P], y is y * silu(z) (the state does not see z).
    """
    x = _f64(x); dt = _f64(dt); A = _f64(A); B = _f64(B); C = _f64(C)
    D = _f64(D); dt_bias = _f64(dt_bias)
    cu = _i32(cu_seqlens)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    S = cu.shape[0] - 1
    assert dt.shape == (T, H) and B.shape == (T, G, N) and C.shape == (T, G, N)
    assert A.shape == (H,)
    cc = _i32(cu_chunk_seqlens)
    K = 0 if cc is None else cc.shape[0] - 1
    init = _f64(initial_states)
    has = None
    if init is not None:
        assert init.shape == (S, H, P, N)
        has = np.ones(S, np.uint8) if has_initial_states is None else \
            np.ascontiguousarray(np.asarray(has_initial_states, dtype=bool), dtype=np.uint8)
    y = np.empty((T, H, P), np.float64)
    cs = np.empty((K, H, P, N), np.float64) if K > 0 else None
    fs = np.empty((S, H, P, N), np.float64)
    rc = _load().oracle_ssd_prefill(
        T, S, H, P, N, G, _ptr(x, ctypes.c_double), _ptr(dt, ctypes.c_double),
        _ptr(B, ctypes.c_double), _ptr(C, ctypes.c_double), _ptr(A, ctypes.c_double),
        _ptr(D, ctypes.c_double), _ptr(dt_bias, ctypes.c_double), int(bool(dt_softplus)),
        float(dt_limit[0]), float(dt_limit[1]), _ptr(cu, ctypes.c_int32), K,
        _ptr(cc, ctypes.c_int32), _ptr(init, ctypes.c_double), _ptr(has, ctypes.c_uint8),
        _ptr(y, ctypes.c_double), _ptr(cs, ctypes.c_double), _ptr(fs, ctypes.c_double),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_ssd_prefill rejected its arguments (code %d)" % rc)
    if z is not None:
        zz = _f64(z)
        assert zz.shape == (T, H, P)
        y = y * silu(zz)
    return y, cs, fs


def chunk_metadata(cu_seqlens, num_computed_tokens, chunk_size):
    """Per-token chunk metadata.

    Returns a dict with int32 arrays ``cu_chunk_seqlens`` [K+1], ``seq_idx``
    [K], ``last_chunk_indices`` [S] (count of chunks of sequences 0..r, minus
    one) and ``chunk_block_col`` [K] (absolute position of the chunk's last
    token // chunk_size).
    """
    cu = _i32(cu_seqlens)
    S = cu.shape[0] - 1
    nc = _i32(num_computed_tokens) if num_computed_tokens is not None else np.zeros(S, np.int32)
    T = int(cu[-1])
    # each sequence adds at most one partial chunk at either end
    max_chunks = min(T, 2 * S + (T + chunk_size - 1) // chunk_size)
    out = {k: np.zeros(n, np.int32) for k, n in (("cu_chunk_seqlens", max_chunks + 1),
                                                ("seq_idx", max_chunks),
                                                ("last_chunk_indices", max(S, 1)),
                                                ("chunk_block_col", max_chunks))}
    K = _load().oracle_chunk_metadata(
        S, int(chunk_size), _ptr(cu, ctypes.c_int32), _ptr(nc, ctypes.c_int32), max_chunks,
        *(_ptr(out[k], ctypes.c_int32) for k in ("cu_chunk_seqlens", "seq_idx",
                                                 "last_chunk_indices", "chunk_block_col")))
    if K < 0:
        raise ValueError("oracle_chunk_metadata rejected its arguments (code %d)" % K)
    return {"cu_chunk_seqlens": out["cu_chunk_seqlens"][:K + 1].copy(),
            "seq_idx": out["seq_idx"][:K].copy(),
            "last_chunk_indices": out["last_chunk_indices"][:S].copy(),
            "chunk_block_col": out["chunk_block_col"][:K].copy()}


def prefill_slots(meta, num_computed_tokens, chunk_size, null_block_id, block_table=None,
                  has_initial_states=None, state_indices=None):
    """Slot routing for prefill, written as plain loops.

    "all" cache mode (``block_table`` [S, cols]): the initial state of r is
    block_table[r, (num_computed[r]-1)//chunk_size] when r has one; chunk k
    stores its end state to block_table[seq_idx[k], chunk_block_col[k]].
    Default mode (``state_indices`` [S]): r's single slot is read as the
    initial state and receives the state of r's last chunk.  Slots equal to
    null_block_id mean "none".  Returns ``(init_slot [S], chunk_slot [K])``.
    """
    seq_idx = meta["seq_idx"]; col = meta["chunk_block_col"]; last = meta["last_chunk_indices"]
    S = len(last); K = len(seq_idx)
    has = [False] * S if has_initial_states is None else [bool(v) for v in has_initial_states]
    nc = [0] * S if num_computed_tokens is None else [int(v) for v in num_computed_tokens]
    init_slot = np.full(S, null_block_id, np.int32)
    chunk_slot = np.full(K, null_block_id, np.int32)
    if block_table is not None:
        bt = np.asarray(block_table)
        for r in range(S):
            if has[r]:
                init_slot[r] = bt[r, (nc[r] - 1) // chunk_size]
        for k in range(K):
            chunk_slot[k] = bt[seq_idx[k], col[k]]
    elif state_indices is not None:
        si = np.asarray(state_indices)
        for r in range(S):
            if has[r]:
                init_slot[r] = si[r]
        for k in range(K):
            r = seq_idx[k]
            if last[r] == k:
                chunk_slot[k] = si[r]
    return init_slot, chunk_slot


def prefill_with_cache(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, init_slot, chunk_slot,
                       null_block_id, cache, D=None, dt_bias=None, dt_softplus=True,
                       dt_limit=(0.0, math.inf), nthreads=None, z=None):
    """Prefill against a state cache ``cache`` [slots,H,P,N] (numpy, any float).

    Every initial state is read before any state is written; chunk end
    states go to their slots unless the slot is null.  Returns ``(y,
    new_cache)``; ``cache`` itself is not modified.
    """
    S = len(init_slot)
    H, P, N = cache.shape[1:]
    init = np.zeros((S, H, P, N), np.float64)
    has = np.zeros(S, bool)
    for r in range(S):
        if int(init_slot[r]) != null_block_id:
            init[r] = cache[int(init_slot[r])]
            has[r] = True
    y, cs, _ = ssd_prefill(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, D=D, dt_bias=dt_bias,
                           initial_states=init, has_initial_states=has,
                           dt_softplus=dt_softplus, dt_limit=dt_limit, nthreads=nthreads, z=z)
    new_cache = np.array(cache, dtype=np.float64, copy=True)
    for k in range(len(chunk_slot)):
        if int(chunk_slot[k]) != null_block_id:
            new_cache[int(chunk_slot[k])] = cs[k]
    return y, new_cache


def ssm_decode(x, dt, A, B, C, read_states, live, D=None, dt_bias=None, dt_softplus=True,
               dt_limit=(0.0, math.inf), nthreads=None, z=None):
    """Decode update for R requests of ``tpr`` tokens each.

    x [R*tpr,H,P], dt [R*tpr,H], B/C [R*tpr,G,N], read_states [R,H,P,N] (the
    state each request resumes from), live [R] booleans.  Token k of request
    r is row r*tpr + k.  Returns ``(y [R*tpr,H,P], states [R,tpr,H,P,N])``
    where states[r,k] is the state right after token k; rows of requests
    that are not live are NaN.  It is the same sequential recurrence as
    prefill, with every token closing a chunk.
    """
    x = _f64(x)
    R = len(live)
    T, H, P = x.shape
    tpr = T // R
    assert tpr * R == T
    N = _f64(B).shape[2]
    cu = np.arange(0, T + 1, tpr, dtype=np.int32)
    cc = np.arange(0, T + 1, dtype=np.int32)
    y, cs, _ = ssd_prefill(x, dt, A, B, C, cu, cc, D=D, dt_bias=dt_bias,
                           initial_states=read_states, has_initial_states=np.ones(R, bool),
                           dt_softplus=dt_softplus, dt_limit=dt_limit, nthreads=nthreads, z=z)
    states = cs.reshape(R, tpr, H, P, N)
    dead = ~np.asarray(live, dtype=bool)
    y = y.reshape(R, tpr, H, P)
    y[dead] = np.nan
    states[dead] = np.nan
    return y.reshape(T, H, P), states


def decode_read_slots(state_indices, num_accepted_tokens, null_block_id):
    """Slot each request resumes from: column num_accepted[r] (0 if absent)."""
    si = np.asarray(state_indices)
    R = si.shape[0]
    out = np.full(R, null_block_id, np.int32)
    for r in range(R):
        a = 0 if num_accepted_tokens is None else int(num_accepted_tokens[r])
        out[r] = si[r, a]
    return out


def decode_with_cache(x, dt, A, B, C, state_indices, num_accepted_tokens, null_block_id, cache,
                      D=None, dt_bias=None, dt_softplus=True, dt_limit=(0.0, math.inf),
                      nthreads=None, z=None):
    """Decode against a cache: rows whose read slot is null are skipped; the
    state after token k goes to column k unless that slot is null.  Reads
    happen before writes.  Returns ``(y, live, new_cache)``."""
    si = np.asarray(state_indices)
    R = si.shape[0]
    T = np.asarray(x).shape[0]
    tpr = T // R
    H, P, N = cache.shape[1:]
    rd = decode_read_slots(si, num_accepted_tokens, null_block_id)
    live = rd != null_block_id
    read = np.zeros((R, H, P, N), np.float64)
    for r in range(R):
        if live[r]:
            read[r] = cache[int(rd[r])]
    y, states = ssm_decode(x, dt, A, B, C, read, live, D=D, dt_bias=dt_bias,
                           dt_softplus=dt_softplus, dt_limit=dt_limit, nthreads=nthreads, z=z)
    new_cache = np.array(cache, dtype=np.float64, copy=True)
    for r in range(R):
        if not live[r]:
            continue
        for k in range(tpr):
            ws = int(si[r, k])
            if ws != null_block_id:
                new_cache[ws] = states[r, k]
    return y, live, new_cache


def causal_conv1d_varlen(xbc, weight, bias, cu_seqlens, init_states=None, has_init=None,
                         activation="silu", cu_chunk_seqlens=None):
    """Depthwise causal conv1d over packed varlen sequences, in fp64.

    The step before the SSM: x, B and C are "hidden_states, B and C after
    depthwise convolution" ("[vllm] vLLM Mamba2 SSD 커널 웜업", the
    MambaMixer2 listing), and each layer keeps a conv state per cache block
    of shape [state_len, conv_dim] ("vLLM v0.20.0 하이브리드 SSM ...", the
    [num_blocks, 3, 3072] conv tensor of "전체 흐름").  Read as Mamba2's
    convolution: for channel c and token t of a sequence,
        out[t, c] = act(bias[c] + sum_k weight[c, k] * in[t - (W-1) + k, c]),
    where the W-1 inputs before the sequence's first token come from its
    conv state (zeros without one) and act is silu or the identity.

    xbc [T, D], weight [D, W], bias [D] or None, cu_seqlens [S+1],
    init_states [S, W-1, D] with has_init [S].  Returns (out [T, D],
    final_states [S, W-1, D], chunk_states [K, W-1, D] or None): the state
    after a token is the last W-1 inputs up to and including it.
    """
    xbc = _f64(xbc)
    w = _f64(weight)
    T, D = xbc.shape
    W = w.shape[1]
    b = np.zeros(D) if bias is None else _f64(bias)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    S = len(cu) - 1
    out = np.empty((T, D))
    final = np.zeros((S, W - 1, D))
    cc = None if cu_chunk_seqlens is None else np.asarray(cu_chunk_seqlens, dtype=np.int64)
    ends = {} if cc is None else {int(cc[k + 1]) - 1: k for k in range(len(cc) - 1)}
    chunk = None if cc is None else np.zeros((len(cc) - 1, W - 1, D))
    for r in range(S):
        a, e = int(cu[r]), int(cu[r + 1])
        hist = np.zeros((W - 1, D))
        if init_states is not None and (has_init is None or has_init[r]):
            hist = _f64(init_states[r]).copy()
        buf = np.concatenate([hist, xbc[a:e]], axis=0)  # inputs W-1 before a, then the sequence
        for i in range(e - a):
            v = b + np.sum(w.T * buf[i:i + W], axis=0)
            out[a + i] = silu(v) if activation == "silu" else v
            k = ends.get(a + i)
            if k is not None:
                chunk[k] = buf[i + 1:i + W]
        final[r] = buf[e - a:e - a + W - 1]
    return out, final, chunk


def causal_conv1d_with_cache(xbc, weight, bias, cu_seqlens, cache, init_slot, out_slot, null_block_id,
                             activation="silu", cu_chunk_seqlens=None, chunk_slot=None):
    """causal_conv1d_varlen against a conv-state cache [slots, W-1, D]: sequence
    r starts from slot init_slot[r] (zeros if null), its final state goes to
    out_slot[r] and each chunk's end state to chunk_slot[k] (unless null);
    every read happens before any write.  Decode is the same call with one
    sequence per request.  Returns (out, new_cache)."""
    S = len(cu_seqlens) - 1
    W1 = cache.shape[1]
    D = cache.shape[2]
    init = np.zeros((S, W1, D))
    has = np.zeros(S, bool)
    for r in range(S):
        s = int(init_slot[r]) if init_slot is not None else null_block_id
        if s != null_block_id:
            init[r] = _f64(cache[s])
            has[r] = True
    out, final, chunk = causal_conv1d_varlen(xbc, weight, bias, cu_seqlens, init, has, activation,
                                             cu_chunk_seqlens)
    new = np.array(cache, dtype=np.float64, copy=True)
    if chunk_slot is not None:
        for k in range(len(chunk_slot)):
            if int(chunk_slot[k]) != null_block_id:
                new[int(chunk_slot[k])] = chunk[k]
    if out_slot is not None:
        for r in range(S):
            if int(out_slot[r]) != null_block_id:
                new[int(out_slot[r])] = final[r]
    return out, new


# ---------------------------------------------------------------- Mamba1 ----
# The selective scan of the Mamba paper (S6) that "[vLLM] Mamba (SSM): 선형 시간
# 복잡도 시퀀스 모델링" summarises in "논문 핵심 내용": every channel d carries
# its own state vector s[d, :] of dstate values with its own decay rates
# A[d, :]; Delta, B and C depend on the token.  Mamba1 has no chunk of its own
# ("[vllm] vLLM Mamba2 SSD 커널 웜업", "vllm/config/model.py 변경 사항": the
# default chunk size becomes 2048); chunks only decide where states are taken
# out for prefix caching, exactly as for Mamba2.


def mamba1_prefill(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens=None, D=None, dt_bias=None,
                   initial_states=None, has_initial_states=None, dt_softplus=True,
                   dt_limit=(0.0, math.inf), nthreads=None, z=None):
    """Sequential fp64 Mamba1 recurrence over packed varlen sequences.

    x and dt [T,Dc], A [Dc,N], B and C [T,G,N], D and dt_bias [Dc],
    initial_states [S,Dc,N].  Returns ``(y [T,Dc], chunk_states [K,Dc,N] or
    None, final_states [S,Dc,N])``; with a gate z [T,Dc], y is y * silu(z).
    """
    x = _f64(x); dt = _f64(dt); A = _f64(A); B = _f64(B); C = _f64(C)
    D = _f64(D); dt_bias = _f64(dt_bias)
    cu = _i32(cu_seqlens)
    T, Dc = x.shape
    G, N = B.shape[1], B.shape[2]
    S = cu.shape[0] - 1
    assert dt.shape == (T, Dc) and B.shape == (T, G, N) and C.shape == (T, G, N) and A.shape == (Dc, N)
    cc = _i32(cu_chunk_seqlens)
    K = 0 if cc is None else cc.shape[0] - 1
    init = _f64(initial_states)
    has = None
    if init is not None:
        assert init.shape == (S, Dc, N)
        has = np.ones(S, np.uint8) if has_initial_states is None else \
            np.ascontiguousarray(np.asarray(has_initial_states, dtype=bool), dtype=np.uint8)
    y = np.empty((T, Dc), np.float64)
    cs = np.empty((K, Dc, N), np.float64) if K > 0 else None
    fs = np.empty((S, Dc, N), np.float64)
    rc = _load().oracle_mamba1_prefill(
        T, S, Dc, N, G, _ptr(x, ctypes.c_double), _ptr(dt, ctypes.c_double), _ptr(B, ctypes.c_double),
        _ptr(C, ctypes.c_double), _ptr(A, ctypes.c_double), _ptr(D, ctypes.c_double),
        _ptr(dt_bias, ctypes.c_double), int(bool(dt_softplus)), float(dt_limit[0]), float(dt_limit[1]),
        _ptr(cu, ctypes.c_int32), K, _ptr(cc, ctypes.c_int32), _ptr(init, ctypes.c_double),
        _ptr(has, ctypes.c_uint8), _ptr(y, ctypes.c_double), _ptr(cs, ctypes.c_double),
        _ptr(fs, ctypes.c_double), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_mamba1_prefill rejected its arguments (code %d)" % rc)
    if z is not None:
        zz = _f64(z)
        assert zz.shape == (T, Dc)
        y = y * silu(zz)
    return y, cs, fs


def mamba1_prefill_with_cache(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, init_slot, chunk_slot,
                              null_block_id, cache, D=None, dt_bias=None, dt_softplus=True,
                              dt_limit=(0.0, math.inf), nthreads=None, z=None):
    """mamba1_prefill against a state cache [slots,Dc,N]: initial states are
    read before any write; chunk end states go to their slots unless null.
    Returns ``(y, new_cache)``."""
    S = len(init_slot)
    Dc, N = cache.shape[1:]
    init = np.zeros((S, Dc, N), np.float64)
    has = np.zeros(S, bool)
    for r in range(S):
        if int(init_slot[r]) != null_block_id:
            init[r] = cache[int(init_slot[r])]
            has[r] = True
    y, cs, _ = mamba1_prefill(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, D=D, dt_bias=dt_bias,
                              initial_states=init, has_initial_states=has, dt_softplus=dt_softplus,
                              dt_limit=dt_limit, nthreads=nthreads, z=z)
    new_cache = np.array(cache, dtype=np.float64, copy=True)
    for k in range(len(chunk_slot)):
        if int(chunk_slot[k]) != null_block_id:
            new_cache[int(chunk_slot[k])] = cs[k]
    return y, new_cache


def mamba1_decode_with_cache(x, dt, A, B, C, state_indices, num_accepted_tokens, null_block_id, cache,
                             D=None, dt_bias=None, dt_softplus=True, dt_limit=(0.0, math.inf),
                             nthreads=None, z=None):
    """Mamba1 decode against a cache [slots,Dc,N], with the routing of
    ``decode_with_cache``: request r resumes from column num_accepted[r] of
    its state-index row, skips if that slot is null, and the state after its
    token k goes to column k unless null.  Returns ``(y, live, new_cache)``;
    y rows of requests that are not live are NaN."""
    si = np.asarray(state_indices)
    R = si.shape[0]
    x64 = _f64(x)
    T, Dc = x64.shape
    tpr = T // R
    assert tpr * R == T
    N = cache.shape[2]
    rd = decode_read_slots(si, num_accepted_tokens, null_block_id)
    live = rd != null_block_id
    read = np.zeros((R, Dc, N), np.float64)
    for r in range(R):
        if live[r]:
            read[r] = cache[int(rd[r])]
    cu = np.arange(0, T + 1, tpr, dtype=np.int32)
    cc = np.arange(0, T + 1, dtype=np.int32)
    y, cs, _ = mamba1_prefill(x64, dt, A, B, C, cu, cc, D=D, dt_bias=dt_bias, initial_states=read,
                              has_initial_states=np.ones(R, bool), dt_softplus=dt_softplus,
                              dt_limit=dt_limit, nthreads=nthreads, z=z)
    states = cs.reshape(R, tpr, Dc, N)
    y = y.reshape(R, tpr, Dc)
    y[~live] = np.nan
    new_cache = np.array(cache, dtype=np.float64, copy=True)
    for r in range(R):
        if not live[r]:
            continue
        for k in range(tpr):
            ws = int(si[r, k])
            if ws != null_block_id:
                new_cache[ws] = states[r, k]
    return y.reshape(T, Dc), live, new_cache
