"""Parity of ssm_decode_update (CUDA, via the C ABI) with the fp64 oracle."""
import pytest
import torch

import selective_state_space_mamba2_gb300 as ssd
from selective_state_space_mamba2_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ssd.build()
    torch.cuda.init()


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("null", [0, -1])
def test_spec_decode_small(dtype, null):
    case = W.decode_case(21, live=5, padded=8, tokens_per_req=3, H=4, P=64, N=128, G=2, num_slots=40,
                         dtype=dtype, device=DEV, null_block_id=null)
    # one live request also skips a write column
    case["state_indices"][2, 1] = null
    before = case["cache"].clone()
    err = _err()
    y = PT.run_decode(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    e_y, e_s, same, tol, nlive = PT.check_decode(case, y, before, case["cache"])
    assert nlive == 5 and e_y <= tol and e_s <= tol and same, (e_y, e_s, same)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_spec_decode_output_gate(dtype):
    """The output gate z on the decode path: y * silu(z) for every token of
    the live requests; states and padded rows as without a gate."""
    case = W.decode_case(22, live=5, padded=8, tokens_per_req=3, H=4, P=64, N=128, G=2, num_slots=40,
                         dtype=dtype, device=DEV, null_block_id=0)
    g = torch.Generator(device=DEV).manual_seed(98)
    z = (3.0 * torch.randn(case["x"].shape, generator=g, device=DEV)).to(dtype)
    before = case["cache"].clone()
    err = _err()
    y = PT.run_decode(case, err=err, z=z)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    e_y, e_s, same, tol, nlive = PT.check_decode(case, y, before, case["cache"], z=z)
    assert nlive == 5 and e_y <= tol and e_s <= tol and same, (e_y, e_s, same)


# dstate 128 with headdim 8 .. 128 runs the fixed-index kernel (one instance per headdim); the
# other sizes, headdim 48 among them, run the general one.
@pytest.mark.parametrize("N,P", [(16, 8), (64, 32), (256, 64), (128, 8), (128, 16), (128, 32), (128, 48),
                                 (128, 128)])
def test_decode_other_state_sizes(N, P):
    case = W.decode_case(22, live=3, padded=4, tokens_per_req=2, H=2, P=P, N=N, G=1, num_slots=12,
                         device=DEV)
    before = case["cache"].clone()
    y = PT.run_decode(case)
    torch.cuda.synchronize()
    e_y, e_s, same, tol, _ = PT.check_decode(case, y, before, case["cache"])
    assert e_y <= tol and e_s <= tol and same


def test_single_token_in_place_update():
    """1 token per request: the read slot is also the write slot."""
    case = W.decode_case(23, live=6, padded=6, tokens_per_req=1, H=4, P=64, N=128, G=4, num_slots=10,
                         device=DEV, spec_accept=False)
    before = case["cache"].clone()
    y = PT.run_decode(case)
    torch.cuda.synchronize()
    e_y, e_s, same, tol, _ = PT.check_decode(case, y, before, case["cache"])
    assert e_y <= tol and e_s <= tol and same


def test_spec_decode_batch_full_size_sampled():
    """256 live requests padded to 512, 1+3 tokens, U{0..3} accepted, in place on
    a [8192,48,64,128] cache: 24 sampled requests (live and padded) checked
    against the oracle on every head; all other slots by fingerprint."""
    case = W.spec_decode_batch(DEV)
    fp_before = PT.slot_fingerprints(case["cache"])
    sample = list(range(0, 256, 16)) + [300, 400, 511, 1, 2, 3, 255, 256]
    si = case["state_indices"]
    rd = [int(si[r, int(case["num_accepted"][r])]) for r in sample]
    before_rows = {s: case["cache"][s].clone() for s in rd if s != case["null_block_id"]}
    err = _err()
    y = PT.run_decode(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    class _View:  # oracle reads only the sampled read slots
        def __getitem__(self, s):
            return before_rows[int(s)]
    e_y, e_s, dead_ok, tol, nlive = PT.check_decode(dict(case), y, _View(), case["cache"], requests=sample,
                                                   check_untouched=False)
    assert nlive == 20 and e_y <= tol and e_s <= tol and dead_ok, (e_y, e_s)
    written = set()
    for r in range(256):
        written.update(int(v) for v in si[r].tolist())
    fp_after = PT.slot_fingerprints(case["cache"])
    mask = torch.ones_like(fp_after, dtype=torch.bool)
    mask[torch.tensor(sorted(written), device=DEV)] = False
    assert torch.equal(fp_after[mask], fp_before[mask])


@pytest.mark.parametrize("N,P", [(16, 16), (128, 64)])
def test_more_tokens_per_request_than_one_staging_batch(N, P):
    """11 tokens per request: the kernels stage a request's tokens 8 at a time, so the state
    carries over from one batch of staged tokens to the next."""
    case = W.decode_case(25, live=3, padded=4, tokens_per_req=11, H=2, P=P, N=N, G=1, num_slots=40,
                         device=DEV)
    before = case["cache"].clone()
    err = _err()
    y = PT.run_decode(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    e_y, e_s, same, tol, nlive = PT.check_decode(case, y, before, case["cache"])
    assert nlive == 3 and e_y <= tol and e_s <= tol and same, (e_y, e_s, same)


@pytest.mark.parametrize("N,P", [(16, 16), (128, 64)])
def test_bad_accepted_column_and_slot_are_reported(N, P):
    case = W.decode_case(24, live=3, padded=3, tokens_per_req=2, H=2, P=P, N=N, G=1, num_slots=10,
                         device=DEV)
    case["num_accepted"][0] = 5
    case["state_indices"][1, 1] = 77
    before = case["cache"].clone()
    err = _err()
    PT.run_decode(case, err=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & ssd.DEVERR_COLUMN and e & ssd.DEVERR_SLOT
    # request 0 skipped entirely: its slots are untouched
    for s in case["state_indices"][0].tolist():
        assert torch.equal(case["cache"][s].view(torch.int32), before[s].view(torch.int32))
