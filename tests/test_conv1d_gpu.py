"""Parity of the depthwise causal conv1d (CUDA, via the C ABI) with the fp64 oracle.

The conv states are exact copies of inputs, so they must match bit for bit;
the outputs are compared with the tolerance of the SSM outputs (2e-2 of the
RMS for bf16, first half ulp excused; 1e-4 for fp32)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_mamba2_gb300 as ssd
from tests import parity as PT

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = 0x7FC0


@pytest.fixture(scope="module", autouse=True)
def _built():
    ssd.build()
    torch.cuda.init()


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _inputs(seed, T, dim_x, dim_bc, W, dtype, slots):
    g = torch.Generator(device="cpu").manual_seed(seed)
    D = dim_x + 2 * dim_bc
    xbc = torch.randn(T, D, generator=g).to(dtype).to(DEV)
    weight = (0.5 * torch.randn(D, W, generator=g)).to(DEV)
    bias = (0.3 * torch.randn(D, generator=g)).to(DEV)
    state = torch.randn(slots, W - 1, D, generator=g).to(dtype).to(DEV)
    return xbc, weight, bias, state


def _check_outputs(xbc_out, want, dim_x, dim_bc, dtype):
    got = torch.cat(xbc_out, dim=1).double().cpu().numpy()
    return PT.y_err(got, want, dtype)


def _mark_unused(state, used):
    """Every slot not in ``used`` gets a NaN bit pattern (bf16: 0x7FC0...), so a stray read shows."""
    mask = torch.ones(state.shape[0], dtype=torch.bool)
    mask[sorted(used)] = False
    idx = mask.nonzero().flatten().to(state.device)
    if state.dtype == torch.bfloat16:
        state.view(torch.int16)[idx] = SENTINEL
    else:
        state.view(torch.int32)[idx] = 0x7FC0DEAD


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [4, 3, 2])
def test_conv1d_varlen_prefix_cached(dtype, W):
    """Ragged packed sequences with unaligned computed prefixes (partial first
    chunks), an empty sequence, sequences shorter than W - 1, mixed initial
    states, conv states stored at every chunk end ("all" cache mode, slots
    from the same block table as the SSM states), and a 256-channel x part
    with 64-channel B and C."""
    new = [300, 1, 0, 2, 129, 64, 517]
    nc = [10, 64, 0, 7, 63, 0, 200]
    has = [True, True, False, True, False, False, True]
    S, Q, dim_x, dim_bc = len(new), 64, 256, 64
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    T = int(cu[-1])
    cols = [(nc[r] + new[r] + Q - 1) // Q + 1 for r in range(S)]
    rng = np.random.default_rng(5)
    slots = 1 + sum(cols) + 8
    perm = rng.permutation(np.arange(1, slots))
    bt = np.zeros((S, max(cols)), np.int32)
    o = 0
    for r in range(S):
        bt[r, :cols[r]] = perm[o:o + cols[r]]
        o += cols[r]
    meta = ssd.ssd_chunk_metadata(cu, Q, nc, has, block_table=bt, null_block_id=0)
    K = int(meta["cu_chunk_seqlens"].shape[0] - 1)
    xbc, weight, bias, state = _inputs(1, T, dim_x, dim_bc, W, dtype, slots)
    init = meta["init_slot"][:S]
    _mark_unused(state, [int(s) for s in init if s != 0])
    before = state.clone()
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(DEV) for k, v in meta.items()}
    err = _err()
    x, B, C = ssd.ssd_conv1d_varlen(xbc, weight, torch.from_numpy(cu).to(DEV), dim_x, dim_bc, bias=bias,
                                    conv_state=state, init_slot=d["init_slot"][:S], chunk_slot=d["chunk_slot"][:K],
                                    cu_chunk_seqlens=d["cu_chunk_seqlens"], last_chunk_indices=d["last_chunk_indices"][:S],
                                    null_block_id=0, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want, new_cache = oracle.causal_conv1d_with_cache(
        xbc.double().cpu().numpy(), weight.double().cpu().numpy(), bias.double().cpu().numpy(), cu,
        before.double().cpu().numpy(), init, None, 0, activation="silu",
        cu_chunk_seqlens=meta["cu_chunk_seqlens"], chunk_slot=meta["chunk_slot"][:K])
    e = _check_outputs((x, B, C), want, dim_x, dim_bc, dtype)
    assert e <= PT.TOL[dtype], e
    written = [int(s) for s in meta["chunk_slot"][:K] if s != 0]
    got = state[torch.tensor(written, device=DEV)].double().cpu().numpy()
    assert np.array_equal(got, new_cache[written]), "a stored conv state differs from its inputs"
    mask = torch.ones(slots, dtype=torch.bool, device=DEV)
    mask[torch.tensor(written, device=DEV)] = False
    bits = torch.int16 if dtype == torch.bfloat16 else torch.int32
    assert torch.equal(state[mask].view(bits), before[mask].view(bits)), "a slot no chunk writes was modified"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("tpr", [1, 2])
def test_conv1d_update_decode_with_padding(dtype, tpr):
    """Decode: each live request continues its slot's conv state for tpr
    tokens and leaves the state after its last token in the same slot;
    padded rows (null slot) are neither read nor written; identity and silu."""
    R, live, dim_x, dim_bc, W = 12, 9, 128, 32, 4
    slots = 40
    rng = np.random.default_rng(6)
    si = np.zeros(R, np.int32)
    si[:live] = rng.permutation(np.arange(1, slots))[:live]
    rng.shuffle(si)
    for act in ("silu", "none"):
        xbc, weight, bias, state = _inputs(2, R * tpr, dim_x, dim_bc, W, dtype, slots)
        _mark_unused(state, [int(s) for s in si if s != 0])
        before = state.clone()
        x_out = torch.full((R * tpr, dim_x), float("nan"), dtype=dtype, device=DEV)
        err = _err()
        x, B, C = ssd.ssd_conv1d_update(xbc, weight, state, torch.from_numpy(si).to(DEV), dim_x, dim_bc,
                                        bias=bias, activation=act, null_block_id=0, x_out=x_out, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        cu = np.arange(0, R * tpr + 1, tpr, dtype=np.int32)
        livereq = si != 0
        want, new_cache = oracle.causal_conv1d_with_cache(
            xbc.double().cpu().numpy(), weight.double().cpu().numpy(), bias.double().cpu().numpy(), cu,
            before.double().cpu().numpy(), si, si, 0, activation=act)
        rows = np.repeat(livereq, tpr)
        got = torch.cat((x, B, C), dim=1).double().cpu().numpy()
        e = PT.y_err(got[rows], want[rows], dtype)
        assert e <= PT.TOL[dtype], (act, e)
        assert np.all(np.isnan(x.double().cpu().numpy()[~rows])), "a padded row was written"
        ws = [int(s) for s in si if s != 0]
        assert np.array_equal(state[torch.tensor(ws, device=DEV)].double().cpu().numpy(), new_cache[ws])
        mask = torch.ones(slots, dtype=torch.bool, device=DEV)
        mask[torch.tensor(ws, device=DEV)] = False
        bits = torch.int16 if dtype == torch.bfloat16 else torch.int32
        assert torch.equal(state[mask].view(bits), before[mask].view(bits))


def test_conv1d_feeds_prefill_unchanged():
    """The conv outputs are ordinary contiguous x [T, H*P], B and C [T, G*N]
    tensors: the SSM prefill run on them (viewed as [T,H,P] and [T,G,N]) gives
    the oracle's SSM output of the oracle's conv output."""
    H, P, N, G, W = 4, 64, 128, 2, 4
    new = [200, 57]
    cu = np.array([0, 200, 257], np.int32)
    T = 257
    xbc, weight, bias, _ = _inputs(3, T, H * P, G * N, W, torch.bfloat16, 2)
    x, B, C = ssd.ssd_conv1d_varlen(xbc, weight, torch.from_numpy(cu).to(DEV), H * P, G * N, bias=bias)
    meta = ssd.ssd_chunk_metadata(cu, 64, None, None, null_block_id=-1)
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(DEV) for k, v in meta.items()}
    K = int(meta["cu_chunk_seqlens"].shape[0] - 1)
    g = torch.Generator(device="cpu").manual_seed(4)
    dt = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
    A = -torch.exp(torch.rand(H, generator=g) * 2).to(DEV)
    Dv = torch.randn(H, generator=g).to(DEV)
    bias_dt = (torch.rand(H, generator=g) * 3 - 4).to(DEV)
    y = ssd.ssd_prefill_varlen(x.view(T, H, P), dt, A, B.view(T, G, N), C.view(T, G, N),
                               torch.from_numpy(cu).to(DEV), d["cu_chunk_seqlens"], d["seq_idx"][:K],
                               d["last_chunk_indices"][:2], D=Dv, dt_bias=bias_dt, null_block_id=-1,
                               chunk_size=64)
    torch.cuda.synchronize()
    conv, _, _ = oracle.causal_conv1d_varlen(xbc.double().cpu().numpy(), weight.double().cpu().numpy(),
                                             bias.double().cpu().numpy(), cu)
    got = torch.cat((x, B, C), dim=1).double().cpu().numpy()
    assert PT.y_err(got, conv, torch.bfloat16) <= PT.TOL[torch.bfloat16]
    # the SSM oracle on the conv outputs exactly as the prefill call read them
    xo = x.double().cpu().numpy().reshape(T, H, P)
    Bo, Co = B.double().cpu().numpy().reshape(T, G, N), C.double().cpu().numpy().reshape(T, G, N)
    yo, _, _ = oracle.ssd_prefill(xo, dt.cpu(), A.cpu(), Bo, Co, cu, meta["cu_chunk_seqlens"], D=Dv.cpu(),
                                  dt_bias=bias_dt.cpu())
    assert PT.y_err(y.double().cpu().numpy(), yo, torch.bfloat16) <= PT.TOL[torch.bfloat16]
