"""Pins for the CPU oracle: each test checks the oracle against something
other than itself -- closed forms, invariants, an independent matrix-form
evaluation, hand-expanded arithmetic, or the chunking loop printed (in part)
on "[vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링", section
"청크 메타데이터 계산"."""
import math

import numpy as np
import pytest

from tests import ssd_forms as F

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_case(rng, T, H, P, N, G, bias=(-4.0, -1.0)):
    x = rng.standard_normal((T, H, P))
    dt = rng.standard_normal((T, H))
    B = rng.standard_normal((T, G, N))
    C = rng.standard_normal((T, G, N))
    A = -np.exp(rng.uniform(0, 2, H))
    D = rng.standard_normal(H)
    dt_bias = rng.uniform(bias[0], bias[1], H)
    return x, dt, A, B, C, D, dt_bias


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sequential_equals_matrix_form_whole_sequence(oracle_lib, seed):
    """Pin 1a: the token-by-token recurrence equals the materialised quadratic
    form y = (L o C B^T) (Delta x) + exp(cs) C h0 + D x on one sequence."""
    rng = np.random.default_rng(seed)
    T, H, P, N, G = 48, 4, 3, 5, 2
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, T, H, P, N, G)
    h0 = rng.standard_normal((1, H, P, N))
    y, _, fs = oracle_lib.ssd_prefill(x, dt, A, B, C, [0, T], D=D, dt_bias=dt_bias,
                                      initial_states=h0)
    yq, endq = F.quadratic_segment(x, F.deltas(dt, dt_bias), A, B, C, D, h0[0])
    assert F.rel_err(y, yq) < 1e-12
    assert F.rel_err(fs[0], endq) < 1e-12


@pytest.mark.parametrize("chunk", [1, 3, 8, 16, 64])
def test_sequential_equals_chunked_evaluation(oracle_lib, chunk):
    """Pin 1b: chunked evaluation (matrix form in each chunk, state passed
    between chunks) equals sequential evaluation at several chunk sizes, on
    packed varlen sequences with and without initial states."""
    rng = np.random.default_rng(100 + chunk)
    lens = [17, 1, 40, 0, 29]
    nc = [5, 0, 3, 0, 70]
    H, P, N, G = 4, 4, 6, 2
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, T, H, P, N, G)
    meta = oracle_lib.chunk_metadata(cu, nc, chunk)
    init = rng.standard_normal((len(lens), H, P, N))
    has = np.array([1, 0, 1, 1, 0], bool)
    y, cs, fs = oracle_lib.ssd_prefill(x, dt, A, B, C, cu, meta["cu_chunk_seqlens"], D=D,
                                       dt_bias=dt_bias, initial_states=init,
                                       has_initial_states=has)
    yc, csc, fsc = F.chunked_prefill(x, dt, A, B, C, D, dt_bias, cu, meta["cu_chunk_seqlens"],
                                     init=[init[r] if has[r] else None for r in range(len(lens))])
    assert F.rel_err(y, yc) < 1e-12
    assert F.rel_err(cs, csc) < 1e-12
    assert F.rel_err(fs, fsc) < 1e-12


def test_A_zero_gives_prefix_sum(oracle_lib):
    """Pin 2: with A = 0 every decay is 1, so the state is h0 plus the running
    sum of Delta_s x_s (outer) B_s, and y_t = C_t . h_t + D x_t."""
    rng = np.random.default_rng(7)
    T, H, P, N, G = 30, 2, 3, 4, 1
    x, dt, _, B, C, D, dt_bias = _rand_case(rng, T, H, P, N, G)
    A = np.zeros(H)
    h0 = rng.standard_normal((1, H, P, N))
    y, _, fs = oracle_lib.ssd_prefill(x, dt, A, B, C, [0, T], D=D, dt_bias=dt_bias,
                                      initial_states=h0)
    d = F.deltas(dt, dt_bias)
    incr = np.einsum("th,thp,tn->thpn", d, x, B[:, 0, :])
    states = h0[0][None] + np.cumsum(incr, axis=0)
    ycf = np.einsum("tn,thpn->thp", C[:, 0, :], states) + D[None, :, None] * x
    assert F.rel_err(y, ycf) < 1e-12
    assert F.rel_err(fs[0], states[-1]) < 1e-12


def test_delta_to_zero_leaves_state(oracle_lib):
    """Pin 3: dt_bias = -100 makes Delta ~ 3.7e-44, so the state stays h0 and
    y = C . h0 + D x."""
    rng = np.random.default_rng(8)
    T, H, P, N, G = 25, 3, 2, 4, 3
    x, dt, A, B, C, D, _ = _rand_case(rng, T, H, P, N, G)
    dt = np.clip(dt, -3, 3)
    dt_bias = np.full(H, -100.0)
    h0 = rng.standard_normal((1, H, P, N))
    y, _, fs = oracle_lib.ssd_prefill(x, dt, A, B, C, [0, T], D=D, dt_bias=dt_bias,
                                      initial_states=h0)
    assert np.max(np.abs(fs[0] - h0[0])) < 1e-30
    yexp = np.einsum("tgn,gpn->tgp", C, h0[0]) + D[None, :, None] * x
    assert F.rel_err(y, yexp) < 1e-14


def test_prefill_then_decode_equals_longer_prefill(oracle_lib):
    """Pin 4: decoding k tokens from the prefill's final state continues the
    same recurrence as one prefill over all tokens."""
    rng = np.random.default_rng(9)
    T0, k, H, P, N, G = 37, 5, 4, 3, 4, 2
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, T0 + k, H, P, N, G)
    y_all, _, fs_all = oracle_lib.ssd_prefill(x, dt, A, B, C, [0, T0 + k], D=D, dt_bias=dt_bias)
    y_pre, _, fs_pre = oracle_lib.ssd_prefill(x[:T0], dt[:T0], A, B[:T0], C[:T0], [0, T0], D=D,
                                              dt_bias=dt_bias)
    y_dec, st = oracle_lib.ssm_decode(x[T0:], dt[T0:], A, B[T0:], C[T0:], fs_pre, [True], D=D,
                                      dt_bias=dt_bias)
    assert F.rel_err(y_pre, y_all[:T0]) < 1e-13
    assert F.rel_err(y_dec, y_all[T0:]) < 1e-13
    assert F.rel_err(st[0, -1], fs_all[0]) < 1e-13
    # one token per decode call, k calls in a row, gives the same
    h = fs_pre
    for i in range(k):
        yi, sti = oracle_lib.ssm_decode(x[T0 + i:T0 + i + 1], dt[T0 + i:T0 + i + 1], A,
                                        B[T0 + i:T0 + i + 1], C[T0 + i:T0 + i + 1], h, [True],
                                        D=D, dt_bias=dt_bias)
        assert F.rel_err(yi, y_all[T0 + i:T0 + i + 1]) < 1e-13
        h = sti[:, 0]


def test_restart_from_chunk_boundary_equals_recompute(oracle_lib):
    """Pin 5: the state stored at a chunk boundary (prefix caching), fed back
    as the initial state with an aligned num_computed, reproduces the rest of
    the full computation."""
    rng = np.random.default_rng(10)
    Q, m, rest, H, P, N, G = 8, 3, 13, 2, 3, 4, 1
    T = Q * m + rest
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, T, H, P, N, G)
    meta = oracle_lib.chunk_metadata([0, T], [0], Q)
    y_full, cs, _ = oracle_lib.ssd_prefill(x, dt, A, B, C, [0, T], meta["cu_chunk_seqlens"], D=D,
                                           dt_bias=dt_bias)
    assert int(meta["chunk_block_col"][m - 1]) == m - 1
    boundary = cs[m - 1]
    meta2 = oracle_lib.chunk_metadata([0, rest], [Q * m], Q)
    y2, cs2, _ = oracle_lib.ssd_prefill(x[Q * m:], dt[Q * m:], A, B[Q * m:], C[Q * m:], [0, rest],
                                        meta2["cu_chunk_seqlens"], D=D, dt_bias=dt_bias,
                                        initial_states=boundary[None])
    assert F.rel_err(y2, y_full[Q * m:]) < 1e-13
    assert F.rel_err(cs2, cs[m:]) < 1e-13
    # the chunk block columns continue where the cached prefix stopped
    assert meta2["chunk_block_col"].tolist() == meta["chunk_block_col"][m:].tolist()


def test_scalar_filter_hand_expanded(oracle_lib):
    """Pin 6: with H = P = N = G = 1 the recurrence is the scalar filter
    h_t = a_t h_{t-1} + b_t; expanded by hand for three tokens."""
    A, D, bias = -0.5, 0.25, 0.3
    dts = [0.2, -1.0, 0.7]
    xs = [1.5, -2.0, 0.5]
    Bs = [0.3, 1.2, -0.8]
    Cs = [2.0, -0.5, 1.1]
    h0 = 0.9
    d = [math.log(1.0 + math.exp(v + bias)) for v in dts]
    a = [math.exp(di * A) for di in d]
    b = [d[i] * xs[i] * Bs[i] for i in range(3)]
    h1 = a[0] * h0 + b[0]
    h2 = a[1] * a[0] * h0 + a[1] * b[0] + b[1]
    h3 = a[2] * a[1] * a[0] * h0 + a[2] * a[1] * b[0] + a[2] * b[1] + b[2]
    yexp = [Cs[0] * h1 + D * xs[0], Cs[1] * h2 + D * xs[1], Cs[2] * h3 + D * xs[2]]
    sh = lambda v: np.array(v, np.float64).reshape(3, 1, 1)
    y, _, fs = oracle_lib.ssd_prefill(sh(xs), np.array(dts).reshape(3, 1), np.array([A]),
                                      sh(Bs), sh(Cs), [0, 3], D=np.array([D]),
                                      dt_bias=np.array([bias]),
                                      initial_states=np.array([[[[h0]]]]))
    assert np.allclose(y.ravel(), yexp, rtol=1e-14, atol=0)
    assert abs(fs.ravel()[0] - h3) < 1e-14


def test_softplus_and_dt_limit_values(oracle_lib):
    """Delta = softplus(dt + bias) then the dt_limit clamp: softplus(0) = ln 2,
    softplus(v) -> v for large v and -> e^v for very negative v."""
    assert abs(oracle_lib.delta(0.0, 0.0) - math.log(2.0)) < 1e-16
    assert abs(oracle_lib.delta(30.0, 0.0) - (30.0 + math.exp(-30.0))) < 1e-13
    assert abs(oracle_lib.delta(-30.0, 0.0) / math.exp(-30.0) - 1.0) < 1e-12
    assert abs(oracle_lib.delta(1.0, -1.0) - math.log(2.0)) < 1e-16
    assert oracle_lib.delta(5.0, 0.0, dt_limit=(0.0, 1.5)) == 1.5
    assert oracle_lib.delta(-5.0, 0.0, dt_limit=(0.1, 1.5)) == 0.1
    assert oracle_lib.delta(-2.0, 0.0, dt_softplus=False, dt_limit=(-math.inf, math.inf)) == -2.0


def test_dt_limit_clamp_matches_matrix_form(oracle_lib):
    rng = np.random.default_rng(12)
    T, H, P, N, G = 20, 2, 3, 4, 1
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, T, H, P, N, G, bias=(-1.0, 1.0))
    lim = (0.2, 0.6)
    y, _, fs = oracle_lib.ssd_prefill(x, dt, A, B, C, [0, T], D=D, dt_bias=dt_bias, dt_limit=lim)
    yq, endq = F.quadratic_segment(x, F.deltas(dt, dt_bias, True, lim), A, B, C, D,
                                   np.zeros((H, P, N)))
    assert F.rel_err(y, yq) < 1e-12 and F.rel_err(fs[0], endq) < 1e-12


def test_heads_use_consecutive_groups(oracle_lib):
    """Reading of the head-to-group map: consecutive heads share a group
    (g = h // (H/G)).  Zeroing group 1's B and C leaves heads 2 and 3 with
    y = D x exactly while heads 0 and 1 still see the state."""
    rng = np.random.default_rng(13)
    T, H, P, N, G = 12, 4, 2, 3, 2
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, T, H, P, N, G)
    B[:, 1] = 0.0
    C[:, 1] = 0.0
    y, _, _ = oracle_lib.ssd_prefill(x, dt, A, B, C, [0, T], D=D, dt_bias=dt_bias)
    for h in (2, 3):
        assert np.array_equal(y[:, h], D[h] * x[:, h])
    for h in (0, 1):
        assert np.max(np.abs(y[:, h] - D[h] * x[:, h])) > 1e-3


def _chunk_loop_from_page(cu_seqlens, num_computed, chunk_size):
    """The chunking loop of the "청크 메타데이터 계산" section, completed in its
    plainest way: first close the unaligned remainder of the previous chunk,
    then full chunks of chunk_size, then a partial tail."""
    cu_chunk = [0]
    seq_idx = []
    last = []
    pos = 0
    for r in range(len(cu_seqlens) - 1):
        nc = int(num_computed[r])
        new = int(cu_seqlens[r + 1]) - int(cu_seqlens[r])
        if nc % chunk_size != 0 and new > 0:
            clen = min(-(-nc // chunk_size) * chunk_size - nc, new)
            pos += clen
            new -= clen
            cu_chunk.append(pos)
            seq_idx.append(r)
        while new > 0:
            clen = min(chunk_size, new)
            pos += clen
            new -= clen
            cu_chunk.append(pos)
            seq_idx.append(r)
        last.append(len(seq_idx) - 1)
    return cu_chunk, seq_idx, last


@pytest.mark.parametrize("seed", range(40))
def test_chunk_metadata_matches_page_loop_and_invariants(oracle_lib, seed):
    rng = np.random.default_rng(1000 + seed)
    S = int(rng.integers(1, 12))
    Q = int(rng.choice([1, 2, 3, 7, 16, 64, 256]))
    lens = rng.integers(0, 5 * Q + 3, S)
    nc = rng.integers(0, 6 * Q + 5, S)
    if seed % 5 == 0:
        nc = (nc // Q) * Q
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    meta = oracle_lib.chunk_metadata(cu, nc, Q)
    cc, si, last = _chunk_loop_from_page(cu, nc, Q)
    assert meta["cu_chunk_seqlens"].tolist() == cc
    assert meta["seq_idx"].tolist() == si
    assert meta["last_chunk_indices"].tolist() == last
    # invariants: each chunk lies in one sequence, holds <= Q tokens, and no
    # chunk crosses an absolute multiple of Q
    for k in range(len(si)):
        a, b = cc[k], cc[k + 1]
        r = si[k]
        assert cu[r] <= a < b <= cu[r + 1] and b - a <= Q
        p0 = int(nc[r]) + a - int(cu[r])
        p1 = int(nc[r]) + b - 1 - int(cu[r])
        assert p0 // Q == p1 // Q == meta["chunk_block_col"][k]
        if b < cu[r + 1]:
            assert (p1 + 1) % Q == 0


def test_prefill_slot_routing_all_mode(oracle_lib):
    """Slot routing in "all" cache mode: the initial state comes from the
    block holding the last computed token; each chunk's end state goes to the
    block of its last token; a partial first chunk shares the block of the
    initial state, which is read before it is overwritten."""
    Q, null = 4, 0
    cu = [0, 6, 9]
    nc = [2, 8]
    meta = oracle_lib.chunk_metadata(cu, nc, Q)
    assert meta["cu_chunk_seqlens"].tolist() == [0, 2, 6, 9]
    bt = np.array([[11, 12, 13, 14], [21, 22, 23, 24]], np.int32)
    init, cslot = oracle_lib.prefill_slots(meta, nc, Q, null, block_table=bt,
                                           has_initial_states=[True, True])
    assert init.tolist() == [11, 22]
    assert cslot.tolist() == [11, 12, 23]
    init_d, cslot_d = oracle_lib.prefill_slots(meta, nc, Q, null, state_indices=[5, 7],
                                               has_initial_states=[False, True])
    assert init_d.tolist() == [null, 7] and cslot_d.tolist() == [null, 5, 7]
    # read-before-write through the cache: sequence 0's init (slot 11) is also
    # chunk 0's output slot
    rng = np.random.default_rng(3)
    H, P, N = 1, 2, 2
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, 9, H, P, N, 1)
    cache = rng.standard_normal((30, H, P, N))
    y, new_cache = oracle_lib.prefill_with_cache(x, dt, A, B, C, cu, meta["cu_chunk_seqlens"],
                                                 init, cslot, null, cache, D=D, dt_bias=dt_bias)
    _, cs, _ = oracle_lib.ssd_prefill(x, dt, A, B, C, cu, meta["cu_chunk_seqlens"], D=D,
                                      dt_bias=dt_bias, initial_states=cache[[11, 22]])
    assert np.array_equal(new_cache[11], cs[0]) and np.array_equal(new_cache[12], cs[1])
    assert np.array_equal(new_cache[23], cs[2])
    untouched = [s for s in range(30) if s not in (11, 12, 23)]
    assert np.array_equal(new_cache[untouched], cache[untouched])


@pytest.mark.parametrize("null", [0, -1])
def test_decode_routing_spec_columns_and_null_rows(oracle_lib, null):
    """Decode routing: request r resumes from column num_accepted[r] of its
    state-index row, writes the state after token k to column k, skips a
    write whose slot is null, and leaves rows whose read slot is null (CUDA
    graph padding) untouched."""
    rng = np.random.default_rng(21)
    H, P, N, G, tpr = 2, 2, 3, 1, 3
    R = 4
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, R * tpr, H, P, N, G)
    si = np.array([[1, 2, 3], [4, 5, null], [null, null, null], [7, 8, 9]], np.int32)
    na = np.array([2, 0, 1, 1], np.int32)
    cache = rng.standard_normal((12, H, P, N))
    y, live, new_cache = oracle_lib.decode_with_cache(x, dt, A, B, C, si, na, null, cache, D=D,
                                                      dt_bias=dt_bias)
    assert live.tolist() == [True, True, False, True]
    # expected from the plain recurrence on each live request
    for r, rd in ((0, 3), (1, 4), (3, 8)):
        rows = slice(r * tpr, (r + 1) * tpr)
        yr, cs, _ = oracle_lib.ssd_prefill(x[rows], dt[rows], A, B[rows], C[rows], [0, tpr],
                                           np.arange(tpr + 1), D=D, dt_bias=dt_bias,
                                           initial_states=cache[rd][None])
        assert np.array_equal(y[rows], yr)
        for k in range(tpr):
            if si[r, k] != null:
                assert np.array_equal(new_cache[si[r, k]], cs[k])
    assert np.all(np.isnan(y[2 * tpr:3 * tpr]))
    written = {1, 2, 3, 4, 5, 7, 8, 9}
    for s in range(12):
        if s not in written:
            assert np.array_equal(new_cache[s], cache[s])


def test_silu_gate_values(oracle_lib):
    """Pin 12a: the oracle's silu equals z * expit(z)
    from scipy and the closed forms silu(0) = 0, silu(ln 3) = (3/4) ln 3
    (sigmoid(ln 3) = 3/4), silu(-ln 3) = -(1/4) ln 3, and silu(z) -> z, -> 0 at
    the two ends."""
    special = pytest.importorskip("scipy.special")
    z = np.linspace(-60.0, 60.0, 2001)
    assert np.allclose(oracle_lib.silu(z), z * special.expit(z), rtol=1e-14, atol=1e-300)
    l3 = math.log(3.0)
    assert oracle_lib.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle_lib.silu(np.array([l3]))[0] - 0.75 * l3) < 1e-15
    assert abs(oracle_lib.silu(np.array([-l3]))[0] + 0.25 * l3) < 1e-15
    assert oracle_lib.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle_lib.silu(np.array([-40.0]))[0]) < 1e-15


def test_gate_scales_output_only(oracle_lib):
    """Pin 12b: a gate z multiplies y elementwise by silu(z) and leaves every
    state untouched; hand-expanded on the scalar filter of pin 6 (two
    tokens), and on a random varlen batch against the ungated run with an
    independently computed z * expit(z)."""
    special = pytest.importorskip("scipy.special")
    A, D, bias, h0 = -0.5, 0.25, 0.3, 0.9
    dts, xs, Bs, Cs, zs = [0.2, -1.0], [1.5, -2.0], [0.3, 1.2], [2.0, -0.5], [0.7, -1.3]
    d = [math.log(1.0 + math.exp(v + bias)) for v in dts]
    h1 = math.exp(d[0] * A) * h0 + d[0] * xs[0] * Bs[0]
    h2 = math.exp(d[1] * A) * h1 + d[1] * xs[1] * Bs[1]
    sig = [1.0 / (1.0 + math.exp(-v)) for v in zs]
    yexp = [(Cs[0] * h1 + D * xs[0]) * zs[0] * sig[0], (Cs[1] * h2 + D * xs[1]) * zs[1] * sig[1]]
    sh = lambda v: np.array(v, np.float64).reshape(2, 1, 1)
    y, _, fs = oracle_lib.ssd_prefill(sh(xs), np.array(dts).reshape(2, 1), np.array([A]), sh(Bs), sh(Cs),
                                      [0, 2], D=np.array([D]), dt_bias=np.array([bias]),
                                      initial_states=np.array([[[[h0]]]]), z=sh(zs))
    assert np.allclose(y.ravel(), yexp, rtol=1e-14, atol=0)
    assert abs(fs.ravel()[0] - h2) < 1e-14
    rng = np.random.default_rng(7)
    T, H, P, N, G = 40, 4, 3, 5, 2
    x, dt, A, B, C, D, dt_bias = _rand_case(rng, T, H, P, N, G)
    z = 3.0 * rng.standard_normal((T, H, P))
    cu, cc = [0, 17, 17, 40], [0, 8, 17, 30, 40]
    y0, cs0, fs0 = oracle_lib.ssd_prefill(x, dt, A, B, C, cu, cc, D=D, dt_bias=dt_bias)
    y1, cs1, fs1 = oracle_lib.ssd_prefill(x, dt, A, B, C, cu, cc, D=D, dt_bias=dt_bias, z=z)
    assert np.array_equal(cs0, cs1) and np.array_equal(fs0, fs1)
    assert np.allclose(y1, y0 * z * special.expit(z), rtol=1e-13, atol=1e-300)


def test_conv1d_equals_numpy_convolve_per_channel(oracle_lib):
    """Pin 13a: without history, the oracle's depthwise causal conv of each
    channel equals numpy's full convolution with the reversed taps, cut to
    the sequence length, plus the bias; with silu it is that value times
    scipy's expit of it; with W = 1 it is the elementwise affine map."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    L, D, W = 23, 5, 4
    x = rng.standard_normal((L, D))
    w = rng.standard_normal((D, W))
    b = rng.standard_normal(D)
    out, final, _ = oracle_lib.causal_conv1d_varlen(x, w, b, [0, L], activation="none")
    ref = np.stack([np.convolve(x[:, c], w[c, ::-1])[:L] + b[c] for c in range(D)], axis=1)
    assert np.allclose(out, ref, rtol=1e-13, atol=1e-13)
    assert np.array_equal(final[0], x[L - W + 1:])
    outs, _, _ = oracle_lib.causal_conv1d_varlen(x, w, b, [0, L], activation="silu")
    assert np.allclose(outs, ref * special.expit(ref), rtol=1e-13, atol=1e-300)
    out1, _, _ = oracle_lib.causal_conv1d_varlen(x, w[:, :1], b, [0, L], activation="none")
    assert np.allclose(out1, x * w[:, 0] + b, rtol=1e-15, atol=1e-15)


def test_conv1d_resume_from_state_and_chunk_states(oracle_lib):
    """Pin 13b: a sequence cut in two, the second part started from the
    first part's final state, gives the outputs and final state of the whole
    (also when a part is shorter than W - 1); the state stored at a chunk end
    is the final state of the prefix ending there; packing sequences
    changes nothing."""
    rng = np.random.default_rng(4)
    D, W = 6, 4
    for L, cut in [(30, 11), (9, 2), (5, 1)]:
        x = rng.standard_normal((L, D))
        w = rng.standard_normal((D, W))
        b = rng.standard_normal(D)
        h0 = rng.standard_normal((1, W - 1, D))
        whole, fw, cs = oracle_lib.causal_conv1d_varlen(x, w, b, [0, L], init_states=h0,
                                                         cu_chunk_seqlens=[0, cut, L])
        p1, f1, _ = oracle_lib.causal_conv1d_varlen(x[:cut], w, b, [0, cut], init_states=h0)
        p2, f2, _ = oracle_lib.causal_conv1d_varlen(x[cut:], w, b, [0, L - cut], init_states=f1)
        assert np.allclose(whole, np.concatenate([p1, p2]), rtol=1e-14, atol=1e-14)
        assert np.array_equal(fw, f2) and np.array_equal(cs[0], f1[0]) and np.array_equal(cs[1], fw[0])
    # packed: two sequences side by side equal two separate calls
    xa, xb = rng.standard_normal((7, D)), rng.standard_normal((12, D))
    w = rng.standard_normal((D, W))
    packed, fp, _ = oracle_lib.causal_conv1d_varlen(np.concatenate([xa, xb]), w, None, [0, 7, 19])
    oa, fa, _ = oracle_lib.causal_conv1d_varlen(xa, w, None, [0, 7])
    ob, fb, _ = oracle_lib.causal_conv1d_varlen(xb, w, None, [0, 12])
    assert np.array_equal(packed, np.concatenate([oa, ob])) and np.array_equal(fp, np.concatenate([fa, fb]))


@pytest.mark.parametrize("null", [0, -1])
def test_conv1d_cache_routing_hand_written(oracle_lib, null):
    """Pin 13c: slot routing of the conv-state cache ("vLLM v0.20.0 하이브리드 SSM
    모델을 위한 분산 서빙 추가", "전체 흐름": one [state_len, conv_dim] conv state
    per cache block), on hand-written slot lists whose expected contents are
    read off the inputs by eye.

    Token t holds 100 (t + 1) + c in channel c, and slot s starts as
    -(10 s + 1 .. 4), so every stored row names where it came from.  W = 3,
    so a state is the last two input rows.  Sequence 0 reads its initial
    state from slot 3 and also writes its final state there (read before
    write); sequence 1 has a null initial slot (zeros); sequence 2 reads slot
    4, which its own first chunk then overwrites; one chunk slot and one
    output slot are null; the slots no one writes keep their bits."""
    W, D = 3, 2
    cu = [0, 5, 6, 9]
    cc = [0, 2, 5, 6, 7, 9]
    x = np.array([[100.0 * (t + 1) + c for c in range(D)] for t in range(9)])
    cache = np.array([[[-(10.0 * s + 1), -(10.0 * s + 2)], [-(10.0 * s + 3), -(10.0 * s + 4)]]
                      for s in range(10)])
    init_slot = [3, null, 4]
    out_slot = [3, 6, null]
    chunk_slot = [7, null, 8, 4, 9]
    w = np.array([[0.5, -1.0, 2.0], [0.25, 3.0, -0.5]])
    b = np.array([0.125, -2.0])
    out, new = oracle_lib.causal_conv1d_with_cache(x, w, b, cu, cache, init_slot, out_slot, null,
                                                   activation="none", cu_chunk_seqlens=cc,
                                                   chunk_slot=chunk_slot)
    want = {
        7: [[100, 101], [200, 201]],      # chunk 0 of sequence 0 ends at token 1
        3: [[400, 401], [500, 501]],      # sequence 0's final state, over its initial slot
        8: [[0, 0], [600, 601]],          # chunk 2 = all of sequence 1, zero history
        6: [[0, 0], [600, 601]],          # sequence 1's final state
        4: [[-43, -44], [700, 701]],      # chunk 3: sequence 2's history row 2, then token 6
        9: [[800, 801], [900, 901]],      # chunk 4
    }
    for s in range(10):
        if s in want:
            assert np.array_equal(new[s], np.array(want[s], np.float64)), s
        else:
            assert np.array_equal(new[s], cache[s]), s
    # outputs: numpy's convolution over [history; tokens] of each sequence, where the
    # history is the hand-chosen slot's original rows (zeros for the null slot)
    hist = [cache[3], np.zeros((2, D)), cache[4]]
    for r in range(3):
        buf = np.concatenate([hist[r], x[cu[r]:cu[r + 1]]])
        L = cu[r + 1] - cu[r]
        ref = np.stack([np.convolve(buf[:, c], w[c, ::-1])[W - 1:W - 1 + L] + b[c] for c in range(D)], axis=1)
        assert np.allclose(out[cu[r]:cu[r + 1]], ref, rtol=1e-15, atol=1e-12), r
