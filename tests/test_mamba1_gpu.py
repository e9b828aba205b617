"""Parity of the Mamba1 selective scan and decode update (CUDA, via the C ABI)
with the fp64 oracle.

Outputs are compared with the SSM tolerance (2e-2 of the RMS for bf16 inputs,
first half ulp excused; 1e-4 for fp32), every state the call writes with the
same bound, and every slot it must not touch bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_mamba2_gb300 as ssd
from selective_state_space_mamba2_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ssd.build()
    torch.cuda.init()


def _np(t):
    return None if t is None else t.double().cpu().numpy()


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _run_scan(c, chunk_size, err=None):
    S = c["cu_seqlens"].numel() - 1
    meta = ssd.ssd_chunk_metadata(c["cu_seqlens"], chunk_size, c["num_computed"], c["has_init"],
                                  block_table=c["block_table"], null_block_id=c["null_block_id"])
    K = int(meta["cu_chunk_seqlens"].shape[0] - 1)
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(DEV) for k, v in meta.items()}
    y = ssd.mamba1_scan_varlen(c["x"], c["dt"], c["A"], c["B"], c["C"], c["cu_seqlens"].to(DEV),
                               d["cu_chunk_seqlens"], d["last_chunk_indices"][:S], D=c["D"], dt_bias=c["dt_bias"],
                               z=c.get("z"), state_cache=c["cache"], init_slot=d["init_slot"][:S],
                               chunk_slot=d["chunk_slot"][:K], null_block_id=c["null_block_id"], err_word=err)
    return y, meta, K


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("N", [16, 8])
@pytest.mark.parametrize("gate", [False, True])
def test_mamba1_scan_varlen_prefix_cached(dtype, N, gate):
    """Ragged packed sequences (an empty one, a single token, lengths that are
    not multiples of the 32/16-token tile), unaligned computed prefixes so the
    first chunk is partial, initial states from the cache for some sequences,
    the state stored at every chunk end through a block table, two groups."""
    new = [300, 1, 0, 77, 513, 64]
    nc = [10, 64, 0, 7, 130, 0]
    has = [True, True, False, True, False, False]
    Q, Dc, G = 64, 256, 2
    c = W.mamba1_prefill_case(11 + N, new, nc, Dc, N, G, Q, dtype=dtype, device=DEV, has_init=has, gate=gate)
    before = c["cache"].clone()
    err = _err()
    y, meta, K = _run_scan(c, Q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    S = len(new)
    want, new_cache = oracle.mamba1_prefill_with_cache(
        _np(c["x"]), _np(c["dt"]), _np(c["A"]), _np(c["B"]), _np(c["C"]), c["cu_seqlens"].numpy(),
        meta["cu_chunk_seqlens"], meta["init_slot"][:S], meta["chunk_slot"][:K], 0, _np(before),
        D=_np(c["D"]), dt_bias=_np(c["dt_bias"]), z=_np(c.get("z")))
    e = PT.y_err(_np(y), want, dtype)
    assert e <= PT.TOL[dtype], (e, PT.where_worst(_np(y), want))
    written = sorted(int(s) for s in meta["chunk_slot"][:K] if s != 0)
    got = c["cache"][torch.tensor(written, device=DEV)].double().cpu().numpy()
    es = PT.rel_err(got, new_cache[written])
    assert es <= PT.TOL[dtype], es
    mask = torch.ones(c["num_slots"], dtype=torch.bool, device=DEV)
    mask[torch.tensor(written, device=DEV)] = False
    assert torch.equal(c["cache"][mask].view(torch.int32), before[mask].view(torch.int32))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("tpr", [1, 3])
@pytest.mark.parametrize("null", [0, -1])
def test_mamba1_state_update_padded_spec(dtype, tpr, null):
    """Decode: 9 live requests padded to 12 with null rows, each resuming from
    the column its num_accepted_tokens names and storing every token's state
    to its own column; padded rows are neither read nor written; with a gate
    for the 3-token case."""
    R, live, Dc, N, G = 12, 9, 128, 16, 1
    c = W.mamba1_decode_case(21 + tpr, live, R, tpr, Dc, N, G, 64, dtype=dtype, device=DEV, null_block_id=null,
                             gate=tpr > 1)
    before = c["cache"].clone()
    si = c["state_indices"]
    y = torch.full_like(c["x"], float("nan"))
    err = _err()
    ssd.mamba1_state_update(c["x"], c["dt"], c["A"], c["B"], c["C"], c["cache"], si.to(DEV),
                            c["num_accepted"].to(DEV), out=y, D=c["D"], dt_bias=c["dt_bias"], z=c.get("z"),
                            null_block_id=null, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want, livem, new_cache = oracle.mamba1_decode_with_cache(
        _np(c["x"]), _np(c["dt"]), _np(c["A"]), _np(c["B"]), _np(c["C"]), si.numpy(), c["num_accepted"].numpy(),
        null, _np(before), D=_np(c["D"]), dt_bias=_np(c["dt_bias"]), z=_np(c.get("z")))
    rows = np.repeat(livem, tpr)
    got = _np(y)
    assert PT.y_err(got[rows], want[rows], dtype) <= PT.TOL[dtype]
    assert np.all(np.isnan(got[~rows])), "a padded row was written"
    written = sorted({int(s) for r in range(R) if livem[r] for s in si[r, :tpr].tolist() if s != null})
    gs = c["cache"][torch.tensor(written, device=DEV)].double().cpu().numpy()
    assert PT.rel_err(gs, new_cache[written]) <= PT.TOL[dtype]
    mask = torch.ones(c["num_slots"], dtype=torch.bool, device=DEV)
    mask[torch.tensor(written, device=DEV)] = False
    assert torch.equal(c["cache"][mask].view(torch.int32), before[mask].view(torch.int32))


def test_mamba1_scan_then_update_continues_the_sequence():
    """The state a prefill leaves at its last chunk end, continued by two
    decode steps on the GPU, matches the oracle's longer prefill."""
    Dc, N, G, Q, L = 128, 16, 1, 2048, 700
    c = W.mamba1_prefill_case(31, [L + 2], [0], Dc, N, G, Q, dtype=torch.float32, device=DEV)
    full = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    pre = dict(c)
    pre["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int32)
    for k in ("x", "dt", "B", "C"):
        pre[k] = c[k][:L].contiguous()
    _, meta, K = _run_scan(pre, Q)
    slot = int(meta["chunk_slot"][K - 1])
    for j in range(2):
        si = torch.tensor([[slot]], dtype=torch.int32, device=DEV)
        yj = ssd.mamba1_state_update(c["x"][L + j:L + j + 1].contiguous(), c["dt"][L + j:L + j + 1].contiguous(),
                                     c["A"], c["B"][L + j:L + j + 1].contiguous(), c["C"][L + j:L + j + 1].contiguous(),
                                     c["cache"], si, D=c["D"], dt_bias=c["dt_bias"])
        torch.cuda.synchronize()
        if j == 1:
            want, _, fs = oracle.mamba1_prefill(_np(full["x"]), _np(full["dt"]), _np(full["A"]), _np(full["B"]),
                                                _np(full["C"]), [0, L + 2], D=_np(full["D"]),
                                                dt_bias=_np(full["dt_bias"]))
            assert PT.rel_err(_np(yj), want[L + 1:]) <= PT.TOL[torch.float32]
            assert PT.rel_err(c["cache"][slot].double().cpu().numpy(), fs[0]) <= PT.TOL[torch.float32]


def test_mamba1_bench_shape_sampled_channels():
    """The benchmark's launch (8 sequences of 8192 tokens, 5120 channels,
    dstate 16, one group, bf16, chunk 2048): channels are independent, so the
    oracle on a sample of 128 channels (two CTAs' worth at each end and in the
    middle) checks those channels' outputs and chunk states exactly."""
    S, L, Dc, N, G, Q = 8, 8192, 5120, 16, 1, 2048
    c = W.mamba1_prefill_case(4, [L] * S, [0] * S, Dc, N, G, Q, dtype=torch.bfloat16, device=DEV,
                              num_slots=S * (L // Q) + 1)
    y, meta, K = _run_scan(c, Q)
    torch.cuda.synchronize()
    ch = np.r_[0:32, 2528:2592, 5088:5120]
    cs = torch.from_numpy(ch).to(DEV)
    sub = lambda t: t[:, cs].contiguous()
    want, cst, _ = oracle.mamba1_prefill(_np(sub(c["x"])), _np(sub(c["dt"])), _np(c["A"][cs]), _np(c["B"]),
                                         _np(c["C"]), c["cu_seqlens"].numpy(), meta["cu_chunk_seqlens"],
                                         D=_np(c["D"][cs]), dt_bias=_np(c["dt_bias"][cs]))
    assert PT.y_err(_np(y[:, cs]), want, torch.bfloat16) <= PT.TOL[torch.bfloat16]
    slots = torch.from_numpy(meta["chunk_slot"][:K].astype(np.int64)).to(DEV)
    got = c["cache"][slots][:, cs].double().cpu().numpy()
    assert PT.rel_err(got, cst) <= PT.TOL[torch.bfloat16]
