"""Parity at the largest sizes the C ABI accepts: a quantised tensor of just under 2^31
elements (the kernels index with 32-bit element offsets) and a GEMM whose A operand is that
large (K = 130944).

The inputs repeat one seeded 128-row block down the rows. Every 128-row tile of the big tensor
then holds the block's values. For MXFP8 the row copy's 1x32 blocks lie within a row and the
column copy's 32-row blocks within a 128-row tile, so the oracle's codes and scales of the
small block are the expected values at every position of the big one, and the GEMM's output
rows repeat with the same period. Sampled rows and columns, including the last ones, are
compared byte for byte (codes, scales) and within the GEMM tolerance (outputs).
"""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, from_dev_bf16, gemm_bf16_close
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F

R_BIG, C_BIG = 16384, 130944           # R * C = 2,145,386,496 < 2^31
PERIOD = 128


def _mx_scale_offsets(rows, kbs, C):
    """Byte offsets of E8M0 scales (row r, 32-block kb) in the tiled layout of a [.][C] copy."""
    r = np.asarray(rows)[:, None]
    kb = np.asarray(kbs)[None, :]
    return ((r >> 7) * (C >> 7) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (kb & 3)


def _big_input(block):
    reps = R_BIG // block.shape[0]
    x = torch.from_numpy(block.view(np.int16)).view(torch.bfloat16).cuda()
    return x.repeat(reps, 1)


@pytest.fixture(scope="module")
def block():
    return bf16_bits_normal(PERIOD, C_BIG, seed=140, outlier_p=1e-4, outlier_factor=40.0)


def test_quantize_mxfp8_largest_tensor(block):
    rec = F.Recipe(kind="mxfp8")
    x = _big_input(block)
    q = F.quantize(rec, x, "activation")
    torch.cuda.synchronize()
    del x
    ref = O.quantize_mxfp8(block)
    rows = [0, 1, 127, 128, 8191, 8320, R_BIG - 129, R_BIG - 1]
    for r in rows:
        assert np.array_equal(q.row[r].cpu().numpy(), ref["row"][r % PERIOD]), r
    kbs = np.arange(C_BIG // 32)
    got = q.row_scale.view(-1)[torch.from_numpy(_mx_scale_offsets(rows, kbs, C_BIG).reshape(-1))
                               .cuda()].cpu().numpy().reshape(len(rows), -1)
    assert np.array_equal(got, ref["row_scale"][np.array(rows) % PERIOD])
    cols = [0, 1, 31, 32, 65535, 65536, C_BIG - 33, C_BIG - 1]
    for c in cols:
        col = q.col[c].cpu().numpy()                     # [R_BIG] codes of source column c
        assert np.array_equal(col.reshape(-1, PERIOD), np.tile(ref["col"][c], (R_BIG // PERIOD, 1))), c
    kbr = np.arange(R_BIG // 32)
    got = q.col_scale.view(-1)[torch.from_numpy(_mx_scale_offsets(cols, kbr, R_BIG).reshape(-1))
                               .cuda()].cpu().numpy().reshape(len(cols), -1)
    want = np.tile(ref["col_scale"][cols], (1, R_BIG // PERIOD))
    assert np.array_equal(got, want)


def test_gemm_mxfp8_largest_operand(block):
    """Y[16384][256] = X W^T with K = 130944: X's quantised row copy is 2.1 GB."""
    rec = F.Recipe(kind="mxfp8")
    N = 256
    wb = bf16_bits_normal(N, C_BIG, seed=141, sigma=0.02)
    x = _big_input(block)
    xq = F.quantize(rec, x, "activation", want_col=False)
    del x
    wq = F.quantize(rec, torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).cuda(),
                    "weight", want_col=False)
    y = F.linear_fwd(rec, xq, wq)
    torch.cuda.synchronize()
    qx = O.quantize_mxfp8(block, want_col=False)
    qw = O.quantize_mxfp8(wb, want_col=False)
    ref = O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]),
                        O.dequant_mx(qw["row"], qw["row_scale"]))
    rows = np.array([0, 127, 128, 8191, R_BIG - 128, R_BIG - 1])
    got = from_dev_bf16(y[torch.from_numpy(rows).cuda()])
    ok, err = gemm_bf16_close(got, ref[rows % PERIOD])
    assert ok, err
