"""CUDA-graph capture of the padded decode step.

"CUDA Graph 지원" on the Mamba (SSM) page pads the decode batch to the graph's
batch size with NULL_BLOCK_ID rows and replays one captured graph.  The decode
calls of this library (the SSM update and the conv update) do no host work
besides their launches and read every size from their arguments, so they can
be captured once on static buffers and replayed with new contents.  These
tests capture both calls with torch's CUDA-graph API, change the tokens, the
slots (including which rows are padding) and the states in place, replay, and
compare with the same calls made eagerly on copies."""
import pytest
import torch

import selective_state_space_mamba2_gb300 as ssd
from selective_state_space_mamba2_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ssd.build()
    torch.cuda.init()


def _decode_step(c, yout, conv, xo, bo, co):
    ssd.ssm_decode_update(c["x"], c["dt"], c["A"], c["B"], c["C"], c["cache"], c["si"], c["na"], out=yout,
                          D=c["D"], dt_bias=c["dt_bias"], null_block_id=0)
    ssd.ssd_conv1d_update(conv["xbc"], conv["w"], conv["state"], conv["si"], 256, 64, bias=conv["b"],
                          null_block_id=0, x_out=xo, B_out=bo, C_out=co)


def _fresh(seed, live):
    c = W.decode_case(seed, live=live, padded=16, tokens_per_req=2, H=4, P=64, N=128, G=2, num_slots=64,
                      device=DEV, null_block_id=0)
    c["si"] = c.pop("state_indices").to(DEV)
    c["na"] = c.pop("num_accepted").to(DEV)
    g = torch.Generator(device=DEV).manual_seed(seed)
    conv = dict(xbc=torch.randn(32, 384, generator=g, device=DEV).to(torch.bfloat16),
                w=0.5 * torch.randn(384, 4, generator=g, device=DEV),
                b=0.3 * torch.randn(384, generator=g, device=DEV),
                state=torch.randn(64, 3, 384, generator=g, device=DEV).to(torch.bfloat16),
                si=c["si"][:, 0].contiguous())
    return c, conv


def test_padded_decode_replays_as_a_graph():
    c, conv = _fresh(31, live=11)
    y = torch.empty_like(c["x"])
    xo = torch.empty(32, 256, dtype=torch.bfloat16, device=DEV)
    bo = torch.empty(32, 64, dtype=torch.bfloat16, device=DEV)
    co = torch.empty(32, 64, dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture (loads the library, sets kernel attributes)
        _decode_step(c, y, conv, xo, bo, co)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _decode_step(c, y, conv, xo, bo, co)
    for seed, live in [(32, 16), (33, 5), (34, 0)]:
        n, nconv = _fresh(seed, live)
        # new contents into the captured buffers, then the same inputs to an eager reference
        for k in ("x", "dt", "B", "C", "cache", "si", "na"):
            c[k].copy_(n[k])
        for k in ("xbc", "state", "si"):
            conv[k].copy_(nconv[k])
        ref = {k: v.clone() for k, v in c.items() if isinstance(v, torch.Tensor)}
        rconv = {k: v.clone() for k, v in conv.items()}
        y.fill_(float("nan"))
        xo.fill_(float("nan"))
        yr = torch.full_like(y, float("nan"))
        xr = torch.full_like(xo, float("nan"))
        br, cr = torch.empty_like(bo), torch.empty_like(co)
        graph.replay()
        _decode_step(ref, yr, rconv, xr, br, cr)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), yr.view(torch.int16)), live
        assert torch.equal(c["cache"].view(torch.int32), ref["cache"].view(torch.int32)), live
        assert torch.equal(xo.view(torch.int16), xr.view(torch.int16)), live
        assert torch.equal(conv["state"].view(torch.int16), rconv["state"].view(torch.int16)), live
