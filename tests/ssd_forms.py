"""Independent fp64 numpy evaluations used to pin the C oracle.

These are written from the matrix (quadratic) form of the selective-SSM
recurrence rather than from its token-by-token update, so a slip in either
one (a dropped term, a transposed state, a wrong decay index) makes the two
disagree.  Test-only code: nothing outside ``tests/`` imports it.
"""
import numpy as np


def softplus(v):
    # log(1 + e^v) via logaddexp, a different route from the C oracle's log1p form
    return np.logaddexp(0.0, v)


def deltas(dt, dt_bias, dt_softplus=True, dt_limit=(0.0, np.inf)):
    v = dt + (0.0 if dt_bias is None else dt_bias[None, :])
    if dt_softplus:
        v = softplus(v)
    return np.clip(v, dt_limit[0], dt_limit[1])


def group_of_heads(H, G):
    return np.repeat(np.arange(G), H // G)


def quadratic_segment(x, delta, A, B, C, D, h0):
    """One segment of tokens with starting state h0 [H,P,N] in matrix form.

    Returns y [L,H,P] and the end state [H,P,N]:
      y[t]  = sum_{s<=t} exp(c_t - c_s) (C_t . B_s) delta_s x_s
              + exp(c_t) C_t . h0 + D x_t,      c = cumsum(delta * A)
      end   = exp(c_L) h0 + sum_s exp(c_L - c_s) delta_s x_s (outer) B_s
    """
    L, H, P = x.shape
    N = B.shape[2]
    G = B.shape[1]
    grp = group_of_heads(H, G)
    y = np.zeros((L, H, P))
    end = np.zeros((H, P, N))
    for h in range(H):
        g = grp[h]
        c = np.cumsum(delta[:, h] * A[h])
        decay = np.exp(c[:, None] - c[None, :])
        mask = np.tril(np.ones((L, L), dtype=bool))
        Lmat = np.where(mask, decay, 0.0)
        CB = C[:, g, :] @ B[:, g, :].T                      # [t, s]
        M = Lmat * CB * delta[None, :, h]                    # [t, s]
        y[:, h, :] = M @ x[:, h, :]
        y[:, h, :] += np.exp(c)[:, None] * (C[:, g, :] @ h0[h].T)
        if D is not None:
            y[:, h, :] += D[h] * x[:, h, :]
        w = np.exp(c[-1] - c) * delta[:, h]                  # [s]
        end[h] = np.exp(c[-1]) * h0[h] + np.einsum("s,sp,sn->pn", w, x[:, h, :], B[:, g, :])
    return y, end


def chunked_prefill(x, dt, A, B, C, D, dt_bias, cu_seqlens, cu_chunk, init=None,
                    dt_softplus=True, dt_limit=(0.0, np.inf)):
    """Chunk-by-chunk evaluation: matrix form inside a chunk, state carried between them."""
    T, H, P = x.shape
    N = B.shape[2]
    delta = deltas(dt, dt_bias, dt_softplus, dt_limit)
    y = np.zeros((T, H, P))
    K = len(cu_chunk) - 1
    chunk_states = np.zeros((K, H, P, N))
    S = len(cu_seqlens) - 1
    final = np.zeros((S, H, P, N))
    k = 0
    for r in range(S):
        s0, s1 = int(cu_seqlens[r]), int(cu_seqlens[r + 1])
        h = np.zeros((H, P, N)) if init is None or init[r] is None else np.array(init[r])
        while k < K and int(cu_chunk[k]) < s1:
            a, b = int(cu_chunk[k]), int(cu_chunk[k + 1])
            assert s0 <= a < b <= s1
            yk, h = quadratic_segment(x[a:b], delta[a:b], A, B[a:b], C[a:b], D, h)
            y[a:b] = yk
            chunk_states[k] = h
            k += 1
        final[r] = h
    return y, chunk_states, final


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    rms = np.sqrt(np.mean(b * b)) if b.size else 0.0
    return float(np.max(np.abs(a - b)) / max(rms, 1e-300)) if a.size else 0.0


def mamba1_quadratic(x, delta, A, B, C, D, h0):
    """Mamba1 (per-channel state) in matrix form, one segment with starting
    state h0 [Dc,N].  For channel d and state index n, with c = A[d,n] *
    cumsum(delta[:, d]):
      s_t[d,n] = sum_{s<=t} exp(c_t - c_s) delta_s[d] B_s[g,n] x_s[d] + exp(c_t) h0[d,n]
      y_t[d]   = sum_n C_t[g,n] s_t[d,n] + D[d] x_t[d]
    Returns y [L,Dc] and the end state [Dc,N]."""
    L, Dc = x.shape
    G, N = B.shape[1], B.shape[2]
    grp = np.repeat(np.arange(G), Dc // G)
    y = np.zeros((L, Dc))
    end = np.zeros((Dc, N))
    mask = np.tril(np.ones((L, L), dtype=bool))
    for d in range(Dc):
        g = grp[d]
        cd = np.cumsum(delta[:, d])
        u = delta[:, d] * x[:, d]
        for n in range(N):
            c = A[d, n] * cd
            decay = np.where(mask, np.exp(c[:, None] - c[None, :]), 0.0)
            s = decay @ (u * B[:, g, n]) + np.exp(c) * h0[d, n]
            y[:, d] += C[:, g, n] * s
            end[d, n] = s[-1]
        if D is not None:
            y[:, d] += D[d] * x[:, d]
    return y, end
