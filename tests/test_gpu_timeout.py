"""Failure detection on the GPU without a fault. A GEMM whose first pipeline stage never becomes
ready, or a quantize (single or grouped) whose first tile never arrives, must come back on its
own with FP8_ERR_TIMEOUT in the caller's status word. The test hooks plant 16 bytes that no
copy delivers. After it, the context is still usable: the next calls on the same stream give
the oracle's results.

Each stalled launch takes about two seconds, the kernel's wait budget. The hook stalls only
the first CTA (pair); the other CTAs, and every later launch, run normally."""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, from_dev_bf16, gemm_bf16_close, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F
    from scaled_quantize_fp8_gb300.binding import linear_fwd_stalled, quantize_stalled

FP8_ERR_TIMEOUT = 6


def _operands(kind, M, N, K, seed):
    rec = F.Recipe(kind=kind)
    xb = bf16_bits_normal(M, K, seed=seed)
    wb = bf16_bits_normal(N, K, seed=seed + 1, sigma=0.02)
    xq = F.quantize(rec, to_dev_bf16(xb), "activation")
    wq = F.quantize(rec, to_dev_bf16(wb), "weight")
    return rec, xb, wb, xq, wq


def _oracle_fprop(kind, xb, wb):
    if kind == "mxfp8":
        qx, qw = O.quantize_mxfp8(xb, want_col=False), O.quantize_mxfp8(wb, want_col=False)
        return O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]),
                             O.dequant_mx(qw["row"], qw["row_scale"]))
    if kind == "tensorwise":
        qx, qw = O.quantize_tensorwise(xb), O.quantize_tensorwise(wb)
        return O.gemm_tn_f64(O.dequant_tensor(qx["row"], qx["scale_inv"]),
                             O.dequant_tensor(qw["row"], qw["scale_inv"]))
    qx, qw = O.quantize_blockwise_1x128(xb), O.quantize_blockwise_128x128(wb)
    return O.gemm_tn_f64(O.dequant_1x128(qx["row"], qx["row_scale_inv"]),
                         O.dequant_128x128(qw["row"], qw["row_scale_inv"]))


# mxfp8: CTA pair with the scale-factor warp (256 x 256 tiles); tensorwise: CTA pair, two
# accumulators; blockwise: single CTA with the per-chunk promotion (128 x 256 tiles)
@pytest.mark.parametrize("kind,M,N,K,tile", [("mxfp8", 256, 256, 512, (256, 256)),
                                              ("tensorwise", 512, 512, 256, (256, 256)),
                                              ("blockwise", 256, 512, 512, (128, 256))])
def test_stalled_gemm_reports_timeout_and_context_survives(kind, M, N, K, tile):
    rec, xb, wb, xq, wq = _operands(kind, M, N, K, seed=120)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    linear_fwd_stalled(rec, xq, wq, y, status)
    torch.cuda.synchronize()                     # returns: the kernel gave up on its own
    assert int(status.item()) == FP8_ERR_TIMEOUT
    # the stalled CTA (pair) has one tile here, its first, which stays zero
    assert not torch.any(y[:tile[0], :tile[1]].view(torch.int16) != 0)

    # the same stream and context still work: a normal GEMM matches the oracle
    status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    y2 = F.linear_fwd(rec, xq, wq, status=status2)
    torch.cuda.synchronize()
    assert int(status2.item()) == 0
    ok, err = gemm_bf16_close(from_dev_bf16(y2), _oracle_fprop(kind, xb, wb))
    assert ok, err


def test_timeout_keeps_the_first_status():
    """The status word keeps the first nonzero code written to it."""
    rec, _, _, xq, wq = _operands("mxfp8", 256, 256, 256, seed=121)
    status = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    y = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    linear_fwd_stalled(rec, xq, wq, y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5


@pytest.mark.parametrize("kind", ["mxfp8", "tensorwise", "delayed", "blockwise"])
def test_stalled_quantize_reports_timeout_and_context_survives(kind):
    rec = F.Recipe(kind=kind)
    R, C = 1024, 512
    xb = bf16_bits_normal(R, C, seed=122)
    x = to_dev_bf16(xb)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = F.empty_qtensor(rec, R, C, "activation")
    quantize_stalled(rec, x, "activation", q, status)
    torch.cuda.synchronize()
    assert int(status.item()) == FP8_ERR_TIMEOUT

    # the next quantize on the same stream is bit-exact
    status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    q2 = F.quantize(rec, x, "activation", status=status2)
    torch.cuda.synchronize()
    assert int(status2.item()) == 0
    if kind == "mxfp8":
        ref = O.quantize_mxfp8(xb)
    elif kind == "tensorwise":
        ref = O.quantize_tensorwise(xb)
    elif kind == "delayed":
        ref = O.DelayedScaling(16).quantize(xb)          # scale 1 from a fresh history
    else:
        ref = O.quantize_blockwise_1x128(xb)
    assert np.array_equal(q2.row.cpu().numpy(), ref["row"])
    assert np.array_equal(q2.col.cpu().numpy(), ref["col"])


@pytest.mark.parametrize("kind", ["mxfp8", "blockwise"])
def test_stalled_quantize_group_reports_timeout_and_context_survives(kind):
    # both instantiations of the grouped kernel: MXFP8, and blockwise (1x128 activation and
    # 128x128 weight in one launch)
    rec = F.Recipe(kind=kind)
    bits = [bf16_bits_normal(1024, 512, seed=123), bf16_bits_normal(512, 256, seed=124)]
    xs = [to_dev_bf16(b) for b in bits]
    roles = ["activation", "weight"]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.quantize_group(rec, xs, roles, status=status, _stalled=True)
    torch.cuda.synchronize()
    assert int(status.item()) == FP8_ERR_TIMEOUT

    # the next grouped call on the same stream is bit-exact
    status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = F.quantize_group(rec, xs, roles, status=status2)
    torch.cuda.synchronize()
    assert int(status2.item()) == 0
    refs = ([O.quantize_mxfp8(b) for b in bits] if kind == "mxfp8" else
            [O.quantize_blockwise_1x128(bits[0]), O.quantize_blockwise_128x128(bits[1])])
    for g, ref in zip(got, refs):
        assert np.array_equal(g.row.cpu().numpy(), ref["row"])
        assert np.array_equal(g.col.cpu().numpy(), ref["col"])
