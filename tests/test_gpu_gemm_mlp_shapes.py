"""GPU parity of the MXFP8 MLP step's four plain-store GEMMs at their own shapes (tokens 8192,
hidden 4096, ffn 16384), in the launch configuration the benchmark times:

    fc2 fprop   y   [8192][4096]  = a . W2^T        K = 16384   a row copy,  W2 row copy
    fc1 dgrad   dX  [8192][4096]  = dh . W1         K = 16384   dh row copy, W1 column copy
    fc2 wgrad   dW2 [4096][16384] = dY^T . a        K = 8192    dY and a column copies
    fc1 wgrad   dW1 [16384][4096] = dh^T . X        K = 8192    dh and X column copies

The GPU quantises seeded bf16 sources (a ~ N(0,1), dh ~ N(0,1e-3) as the backward pass's
gradient, W ~ N(0,0.02)) and runs each GEMM in bf16 and in fp32 output mode. The oracle
quantises the same sources itself, but only the rows of each operand copy that a sample of
the output needs: the first and last 128 output rows and columns plus 64 random ones of each.
A row of a column-wise copy is a column of the source, quantised in 1x32 blocks along the
source's rows, so the oracle quantises the transposed source columns. Checked: bf16 outputs
elementwise within 1e-2 (floor 1e-3 of the sample's max), fp32 outputs normwise within 1e-5
of the fp64 sum, the accumulation-agreement bound at K = 16384 and 8192.
"""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, gemm_bf16_close, gemm_f32_normwise, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F

TOKENS, HIDDEN, FFN = 8192, 4096, 16384

# seeded sources of the step's GEMM operands: shape, sigma, stream
SOURCES = {"x": ((TOKENS, HIDDEN), 1.0, 0), "w1": ((FFN, HIDDEN), 0.02, 1),
           "w2": ((HIDDEN, FFN), 0.02, 3), "dy": ((TOKENS, HIDDEN), 1e-3, 2),
           "a": ((TOKENS, FFN), 1.0, 6), "dh": ((TOKENS, FFN), 1e-3, 7)}
ROLES = {"x": "activation", "a": "activation", "w1": "weight", "w2": "weight", "dy": "grad",
         "dh": "grad"}

# name: (A source and copy, B source and copy, M, N, K)
CASES = {
    "fc2_fprop": (("a", "row"), ("w2", "row"), TOKENS, HIDDEN, FFN),
    "fc1_dgrad": (("dh", "row"), ("w1", "col"), TOKENS, HIDDEN, FFN),
    "fc2_wgrad": (("dy", "col"), ("a", "col"), HIDDEN, FFN, TOKENS),
    "fc1_wgrad": (("dh", "col"), ("x", "col"), FFN, HIDDEN, TOKENS),
}

_SRC = {}


def _source(name):
    if name not in _SRC:
        (r, c), sigma, stream = SOURCES[name]
        _SRC[name] = bf16_bits_normal(r, c, seed=0, stream=stream, sigma=sigma)
    return _SRC[name]


def _sample(n, seed):
    g = np.random.default_rng(seed)
    idx = np.concatenate([np.arange(128), np.arange(n - 128, n), g.choice(n, 64, replace=False)])
    return np.unique(idx)


def _oracle_rows(src, copy, idx):
    """Dequantised rows `idx` of the oracle's row or column copy of a bf16 source (float64)."""
    part = src[idx] if copy == "row" else np.ascontiguousarray(src[:, idx].T)
    q = O.quantize_mxfp8(part, want_col=False)
    return O.dequant_mx(q["row"], q["row_scale"])


def _gpu(name, fp32):
    rec = F.Recipe(kind="mxfp8")
    (an, _), (bn, _), _, _, _ = CASES[name]
    q = {n: F.quantize(rec, to_dev_bf16(_source(n)), ROLES[n]) for n in {an, bn}}
    if name == "fc2_fprop":
        return F.linear_fwd(rec, q["a"], q["w2"], fp32=fp32)
    if name == "fc1_dgrad":
        return F.linear_bwd(rec, q["dh"], None, q["w1"], want_dw=False, fp32=fp32)[0]
    if name == "fc2_wgrad":
        return F.linear_bwd(rec, q["dy"], q["a"], None, want_dx=False, fp32=fp32)[1]
    return F.linear_bwd(rec, q["dh"], q["x"], None, want_dx=False, fp32=fp32)[1]


@pytest.mark.parametrize("name", sorted(CASES))
def test_mlp_step_gemm_sampled(name):
    (an, ac), (bn, bc), M, N, K = CASES[name]
    rows, cols = _sample(M, 21), _sample(N, 22)
    ri, ci = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    got = {}
    for fp32 in (False, True):
        d = _gpu(name, fp32)
        assert tuple(d.shape) == (M, N)
        got[fp32] = d[ri][:, ci].contiguous()
        del d
    torch.cuda.synchronize()
    ref = O.gemm_tn_f64(_oracle_rows(_source(an), ac, rows), _oracle_rows(_source(bn), bc, cols))
    assert ref.shape == (rows.size, cols.size)
    ok, err = gemm_bf16_close(got[False].view(torch.int16).cpu().numpy().view(np.uint16), ref)
    assert ok, (name, "bf16", err)
    ok, err = gemm_f32_normwise(got[True].cpu().numpy(), ref)
    assert ok, (name, "fp32 accumulation", err)
