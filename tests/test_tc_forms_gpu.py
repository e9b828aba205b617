"""The tensor-core operand forms of the fused prefill kernel (TMA tiles with
128-byte swizzle, K-major and MN-major shared-memory descriptors, an A
operand in TMEM) reproduce plain matrix products of the same bf16 values."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _build_probe():
    src = os.path.join(HERE, "tc_probe", "tc_probe.cu")
    out = os.path.join(HERE, "tc_probe", "_build", "libtc_probe.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                               "-Xcompiler", "-fPIC", "-shared", "-I", os.path.join(ROOT, "include"), "-I",
                               os.path.join(ROOT, "selective_state_space_mamba2_gb300", "csrc"), "-o", out, src])
    return ctypes.CDLL(out)


def test_tensor_core_forms_match_matmul():
    lib = _build_probe()
    g = torch.Generator(device="cuda").manual_seed(0)
    r = lambda *s: torch.randn(*s, generator=g, device="cuda").to(torch.bfloat16)
    C, B, X, H, W, P = r(128, 128), r(128, 128), r(128, 64), r(128, 64), r(128, 64), r(128, 128)
    outs = [torch.full((128, 128), float("nan"), device="cuda")] + \
        [torch.full((128, 64), float("nan"), device="cuda") for _ in range(4)] + \
        [torch.full((128, 128), float("nan"), device="cuda")]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.tc_probe_run(p(C), p(B), p(X), p(H), p(W), p(P), *[p(o) for o in outs], p(status),
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and int(status.item()) == 0
    d = lambda t: t.double()
    want = [d(C) @ d(B).T, d(P) @ d(X), d(C) @ d(H), d(B).T @ d(W), None, d(C) @ torch.cat([d(H), d(W)], 1)]
    names = ["C.B^T (SS, K/K)", "P.X (TS, MN B)", "C.H (SS, K A, MN B)", "B^T.W (SS, MN A, MN B)", None,
             "C.[H|W] (SS, K A, MN B, N=128)"]
    errs = [float((d(o) - w).abs().max() / w.abs().max()) for o, w in zip(outs, want) if w is not None]
    names = [n for n in names if n is not None]
    swapped = float((d(outs[4]) - want[3]).abs().max() / want[3].abs().max())
    msg = "; ".join("%s %.2e" % (n, e) for n, e in zip(names, errs)) + "; B^T.W swapped offsets %.2e" % swapped
    print(msg)
    assert all(e < 1e-4 for e in errs), msg
