"""Why the fused prefill rounds its tensor-core operands to fp16 and not bf16.

The kernel's block arithmetic (128-token blocks: S = C B^T, P = fp16(decay . delta . S), Y1 = P X,
Y2 = C Hprev^T with the carried state rounded for the product, dS = (w x)^T B with w x rounded,
fp32 accumulation and an fp32 state) is emulated here on the CPU with the rounded operands in
fp16, as the kernel does, and in bf16, and both are held to the fp64 oracle by the parity
tests' measure (largest error over the output's RMS, bar 2e-2).  fp16 operands stay well inside
the bar; the state's products in bf16 (w x for the state, the carried state for y) do not: the
B and C copies the prep kernel writes are the price of meeting it."""
import math

import numpy as np
import torch

import oracle
from selective_state_space_mamba2_gb300 import workloads as W

BAR = 2e-2


def _emulate(case, op_dtype, Q=128):
    x, dt, A = case["x"].float(), case["dt"].float(), case["A"].float()
    B, C, D, bias = case["B"].float(), case["C"].float(), case["D"].float(), case["dt_bias"].float()
    T, H, P = x.shape
    G = B.shape[1]
    delta = torch.nn.functional.softplus(dt + bias[None])
    y = torch.zeros(T, H, P)
    finals = []
    for h in range(H):
        g = h // (H // G)
        st = torch.zeros(P, B.shape[2])
        for b0 in range(0, T, Q):
            b1 = min(b0 + Q, T)
            L = b1 - b0
            d = delta[b0:b1, h]
            c = torch.cumsum(d * A[h], 0)
            Cb, Bb = C[b0:b1, g], B[b0:b1, g]
            S = Cb @ Bb.T
            Pm = torch.where(torch.tril(torch.ones(L, L, dtype=torch.bool)),
                             torch.exp(c[:, None] - c[None, :]) * d[None, :] * S, torch.zeros(()))
            Pm = (Pm + torch.diag(torch.full((L,), float(D[h])))).half().float()  # P is fp16 in both
            Y1 = Pm @ x[b0:b1, h].half().float()
            Y2 = Cb @ st.to(op_dtype).float().T
            y[b0:b1, h] = Y1 + torch.exp(c)[:, None] * Y2
            wx = ((torch.exp(c[-1] - c) * d)[:, None] * x[b0:b1, h]).to(op_dtype).float()
            st = torch.exp(c[-1]) * st + wx.T @ Bb
        finals.append(st)
    return y, torch.stack(finals)


def _errors(case, op_dtype):
    yo, _, fo = oracle.ssd_prefill(case["x"], case["dt"], case["A"], case["B"], case["C"], case["cu_seqlens"],
                                   None, D=case["D"], dt_bias=case["dt_bias"])
    y, st = _emulate(case, op_dtype)
    ey = float(np.max(np.abs(y.double().numpy() - yo))) / math.sqrt(float(np.mean(yo * yo)))
    fo = np.asarray(fo)[0]
    es = float(np.max(np.abs(st.double().numpy() - fo))) / math.sqrt(float(np.mean(fo * fo)))
    return ey, es


def test_fp16_operands_meet_the_bar_and_bf16_ones_do_not():
    case = W.prefill_case(1, [2048], [0], 4, 64, 128, 1, 256)
    ey16, es16 = _errors(case, torch.float16)
    ey_bf, es_bf = _errors(case, torch.bfloat16)
    assert ey16 <= BAR and es16 <= BAR / 2, (ey16, es16)
    assert es_bf > BAR, es_bf  # the state's products in bf16 miss the bar
