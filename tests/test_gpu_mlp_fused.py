"""GPU parity of the fused MLP steps (MXFP8): fc1 with the GeLU step in the GEMM epilogue
(h's FP8 row copy plus a = gelu(h) as row and column copies, h never stored in bf16), and the
dgrad of fc2 with the GeLU backward in the epilogue (dh = da * gelu'(h) as row and column
copies, da never stored).

Each fused output is checked stage by stage:
- byte for byte against the unfused GPU steps (GEMM storing bf16, then the standalone GeLU /
  dGeLU kernel): both round the same fp32 accumulator to bf16 and apply the same fp32 GeLU;
- the quantisation stage exactly: the oracle's MXFP8 quantiser applied to the GPU's own bf16
  quantiser input (h from the plain GEMM, a and dh from the standalone kernels' bf16 outputs)
  must give every code and every E8M0 byte of both copies;
- the bf16 stages against the oracle's own: h from the oracle's fp64 GEMM and a = gelu(h) from
  its fp64 GeLU agree within one bf16 unit in the last place (the GPU accumulates and
  evaluates in fp32). The fraction of elements one ulp apart is reported, not graded.
"""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, from_dev_bf16, gemm_bf16_close, mx_untile, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _np(t):
    return t.cpu().numpy()


def _check_mx_exact(codes, scale_plain, gpu_in):
    """codes [R][C] and plain E8M0 scales [R][C/32] that the GPU produced from its bf16 tensor
    gpu_in must equal the oracle's MXFP8 quantisation of that same tensor, on every block."""
    ref = O.quantize_mxfp8(gpu_in, want_col=False)
    assert np.array_equal(codes, ref["row"])
    assert np.array_equal(scale_plain, ref["row_scale"])


def _ulp_diff(a_bits, b_bits):
    """Distance in bf16 units in the last place (NaN positions excluded by the caller)."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)


def _within_one_ulp(gpu_bits, ref_bits):
    """The GPU's bf16 stage output against the oracle's: NaN where the oracle has NaN, else at
    most one ulp apart. Returns the fraction of elements that are one ulp apart (diagnostic)."""
    nan = np.isnan(O.bf16_to_f32(ref_bits))
    assert np.array_equal(np.isnan(O.bf16_to_f32(gpu_bits)), nan)
    d = _ulp_diff(gpu_bits[~nan], ref_bits[~nan])
    assert d.size == 0 or int(d.max()) <= 1
    return float(np.mean(d == 1)) if d.size else 0.0


def _check_copies(q, gpu_bf16, M, N, rows=None):
    """Both MXFP8 copies of the [M][N] tensor q against the oracle's quantisation of the GPU's
    bf16 tensor; `rows` (whole 32-row blocks) restricts the check to those token rows."""
    if rows is None:
        rows = np.arange(M)
    _check_mx_exact(_np(q.row)[rows], mx_untile(_np(q.row_scale), M, N)[rows], gpu_bf16[rows])
    if q.col is not None:
        blocks = np.unique(rows // 32)
        assert np.array_equal(np.sort(rows), np.concatenate([np.arange(32 * b, 32 * b + 32)
                                                             for b in blocks]))
        col, cs = _np(q.col), mx_untile(_np(q.col_scale), N, M)
        cols = np.concatenate([np.arange(32 * b, 32 * b + 32) for b in blocks])
        # the column copy's blocks run along the tokens: quantise the transposed token rows
        _check_mx_exact(np.ascontiguousarray(col[:, cols]), np.ascontiguousarray(cs[:, blocks]),
                        np.ascontiguousarray(gpu_bf16[cols].T))


def _same_qtensor(a, b, fields):
    for f in fields:
        x, y = getattr(a, f), getattr(b, f)
        assert torch.equal(x, y), f


def _fc1(M, N, K, seed):
    rec = F.Recipe(kind="mxfp8")
    xb = bf16_bits_normal(M, K, seed=seed, stream=0)
    wb = bf16_bits_normal(N, K, seed=seed, stream=1, sigma=0.02)
    xq = F.quantize(rec, to_dev_bf16(xb), "activation")
    wq = F.quantize(rec, to_dev_bf16(wb), "weight")
    return rec, xb, wb, xq, wq


# the last shape runs 160 pair tiles on the 76 pairs of a full GPU (a partial last round),
# grouped along M (M < N)
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 256, 256), (384, 512, 256),
                                   (512, 384, 512), (256, 128, 384), (2560, 4096, 256)])
def test_fc1_gelu_fused(M, N, K):
    rec, xb, wb, xq, wq = _fc1(M, N, K, seed=M + N)
    a_q, h_q = F.linear_fwd_gelu(rec, xq, wq)
    # unfused GPU steps
    h = F.linear_fwd(rec, xq, wq)
    a_u, h_u, a_bf16 = F.gelu_quantize(rec, h, want_a_bf16=True)
    torch.cuda.synchronize()
    _same_qtensor(a_q, a_u, ("row", "row_scale", "col", "col_scale"))
    _same_qtensor(h_q, h_u, ("row", "row_scale"))
    # GEMM stage: the GPU's bf16 h against the oracle's fp64 sum
    qx, qw = O.quantize_mxfp8(xb, want_col=False), O.quantize_mxfp8(wb, want_col=False)
    h_g, a_g = from_dev_bf16(h), from_dev_bf16(a_bf16)
    ok, err = gemm_bf16_close(h_g, O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]),
                                                 O.dequant_mx(qw["row"], qw["row_scale"])))
    assert ok, err
    # GeLU stage on the same h, then the quantisation of h and a: every byte
    _within_one_ulp(a_g, O.gelu_bf16(h_g))
    _check_copies(h_q, h_g, M, N)
    _check_copies(a_q, a_g, M, N)


# the last shape runs 96 pair tiles (two rounds) in the exchanged tile order (M > N)
@pytest.mark.parametrize("M,Fd,H", [(128, 256, 128), (256, 256, 256), (384, 512, 256),
                                    (512, 384, 128), (4096, 1536, 256)])
def test_fc2_dgrad_dgelu_fused(M, Fd, H):
    rec = F.Recipe(kind="mxfp8")
    seed = M + Fd
    hb = bf16_bits_normal(M, Fd, seed=seed, stream=0, sigma=2.0)
    dyb = bf16_bits_normal(M, H, seed=seed, stream=2, sigma=1e-3)
    w2b = bf16_bits_normal(H, Fd, seed=seed, stream=3, sigma=0.02)
    _, h_q, _ = F.gelu_quantize(rec, to_dev_bf16(hb))      # h's FP8 copy from a seeded h
    dyq = F.quantize(rec, to_dev_bf16(dyb), "grad")
    w2q = F.quantize(rec, to_dev_bf16(w2b), "weight")
    dh_q = F.linear_dgrad_dgelu(rec, dyq, w2q, h_q)
    da, _ = F.linear_bwd(rec, dyq, None, w2q, want_dw=False)
    dh_u, dh_bf16 = F.dgelu_quantize(rec, da, h_q, want_dh_bf16=True)
    torch.cuda.synchronize()
    _same_qtensor(dh_q, dh_u, ("row", "row_scale", "col", "col_scale"))
    # h's FP8 copy from the seeded h, every byte
    qh = O.quantize_mxfp8(hb, want_col=False)
    assert np.array_equal(_np(h_q.row), qh["row"])
    # GEMM stage: da = dY . (W2^T)^T from the column copy of W2, against the fp64 sum
    qdy = O.quantize_mxfp8(dyb, want_col=False)
    qw2t = O.quantize_mxfp8(np.ascontiguousarray(w2b.T), want_col=False)
    da_g = from_dev_bf16(da)
    ok, err = gemm_bf16_close(da_g, O.gemm_tn_f64(O.dequant_mx(qdy["row"], qdy["row_scale"]),
                                                  O.dequant_mx(qw2t["row"], qw2t["row_scale"])))
    assert ok, err
    # dGeLU stage on the same da and FP8 h, then dh's quantisation: every byte
    dh_g = from_dev_bf16(dh_bf16)
    _within_one_ulp(dh_g, O.dgelu_bf16(da_g, qh["row"], qh["row_scale"]))
    _check_copies(dh_q, dh_g, M, Fd)


def test_fc2_dgrad_dgelu_fused_wide_scales():
    """h blocks spread over many MXFP8 scales (tiny, ordinary, large), plus zero, Inf and NaN
    blocks: the epilogue's per-block gelu' table rows and its direct path for blocks outside
    them must give the unfused kernels' bytes, and the oracle's where dh is finite."""
    rec = F.Recipe(kind="mxfp8")
    M, Fd, H = 256, 512, 256
    hb = bf16_bits_normal(M, Fd, seed=61, stream=0, sigma=1.0)
    h = O.bf16_to_f32(hb).reshape(M, Fd // 32, 32).astype(np.float64)
    factors = np.array([2.0 ** -30, 2.0 ** -20, 2.0 ** -12, 1e-3, 1.0, 4.0, 2.0 ** 6, 2.0 ** 9,
                        2.0 ** 14, 2.0 ** 40])
    h *= factors[np.arange(M * (Fd // 32)).reshape(M, Fd // 32) % len(factors)][:, :, None]
    h[3, 5, :] = 0.0
    h[7, 2, 4] = np.inf
    h[9, 1, 7] = np.nan
    h[11, 3, 0] = -np.inf
    hb = O.f64_to_bf16(h.reshape(M, Fd))
    dyb = bf16_bits_normal(M, H, seed=62, stream=2, sigma=1e-3)
    w2b = bf16_bits_normal(H, Fd, seed=63, stream=3, sigma=0.02)
    _, h_q, _ = F.gelu_quantize(rec, to_dev_bf16(hb))
    dyq = F.quantize(rec, to_dev_bf16(dyb), "grad")
    w2q = F.quantize(rec, to_dev_bf16(w2b), "weight")
    dh_q = F.linear_dgrad_dgelu(rec, dyq, w2q, h_q)
    da, _ = F.linear_bwd(rec, dyq, None, w2q, want_dw=False)
    dh_u, dh_bf16 = F.dgelu_quantize(rec, da, h_q, want_dh_bf16=True)
    torch.cuda.synchronize()
    _same_qtensor(dh_q, dh_u, ("row", "row_scale", "col", "col_scale"))
    qh = O.quantize_mxfp8(hb, want_col=False)
    assert np.array_equal(_np(h_q.row), qh["row"])
    sc = mx_untile(_np(h_q.row_scale), M, Fd)
    assert np.array_equal(sc, qh["row_scale"])
    assert sc.min() < 110 and 126 <= sc[sc < 255].max() and (sc == 255).any()
    qdy = O.quantize_mxfp8(dyb, want_col=False)
    qw2t = O.quantize_mxfp8(np.ascontiguousarray(w2b.T), want_col=False)
    da_g = from_dev_bf16(da)
    ok, err = gemm_bf16_close(da_g, O.gemm_tn_f64(O.dequant_mx(qdy["row"], qdy["row_scale"]),
                                                  O.dequant_mx(qw2t["row"], qw2t["row_scale"])))
    assert ok, err
    dh_r = O.dgelu_bf16(da_g, qh["row"], qh["row_scale"])
    dh_g = from_dev_bf16(dh_bf16)
    _within_one_ulp(dh_g, dh_r)
    # NaN blocks of dh (from the Inf / NaN h blocks): codes and scale marked NaN on both sides,
    # and every block, NaN or not, quantised exactly as the oracle quantises the GPU's dh
    nan_r = np.isnan(O.bf16_to_f32(dh_r)).reshape(M, Fd // 32, 32).any(axis=2)
    assert np.array_equal(nan_r, (mx_untile(_np(dh_q.row_scale), M, Fd) == 255))
    _check_copies(dh_q, dh_g, M, Fd)


def _mlp_fused(M, H, Fd, seed):
    """The whole MXFP8 MLP block through the fused steps, final GEMM outputs against the oracle
    run end to end on the same seeded inputs.

    End to end the two sides do not quantise identical tensors: where the GPU's h is one bf16
    ulp off the oracle's, its E4M3 code can move by one step, and gelu'(h), dh and both GEMMs
    behind them follow. The per-element GEMM bound does not cover that, so the end-to-end check
    is normwise, max|C - R| <= 1e-2 max|R| per output; each stage has its own exact check."""
    rec = F.Recipe(kind="mxfp8")
    xb = bf16_bits_normal(M, H, seed=seed, stream=0)
    w1b = bf16_bits_normal(Fd, H, seed=seed, stream=1, sigma=0.02)
    w2b = bf16_bits_normal(H, Fd, seed=seed, stream=3, sigma=0.02)
    dyb = bf16_bits_normal(M, H, seed=seed, stream=2, sigma=1e-3)
    xq = F.quantize(rec, to_dev_bf16(xb), "activation")
    w1q = F.quantize(rec, to_dev_bf16(w1b), "weight")
    w2q = F.quantize(rec, to_dev_bf16(w2b), "weight")
    a_q, h_q = F.linear_fwd_gelu(rec, xq, w1q)
    y = F.linear_fwd(rec, a_q, w2q)
    dyq = F.quantize(rec, to_dev_bf16(dyb), "grad")
    _, dw2 = F.linear_bwd(rec, dyq, a_q, w2q, want_dx=False)
    dh_q = F.linear_dgrad_dgelu(rec, dyq, w2q, h_q)
    dx, dw1 = F.linear_bwd(rec, dh_q, xq, w1q)
    torch.cuda.synchronize()
    qx, qw1, qw2, qdy = (O.quantize_mxfp8(b) for b in (xb, w1b, w2b, dyb))
    dq = lambda q, c: O.dequant_mx(q[c], q[c + "_scale"])  # noqa: E731
    h_r = O.f64_to_bf16(O.gemm_tn_f64(dq(qx, "row"), dq(qw1, "row")))
    qh = O.quantize_mxfp8(h_r, want_col=False)
    qa = O.quantize_mxfp8(O.gelu_bf16(h_r))
    y_r = O.gemm_tn_f64(dq(qa, "row"), dq(qw2, "row"))
    da_r = O.f64_to_bf16(O.gemm_tn_f64(dq(qdy, "row"), dq(qw2, "col")))
    dw2_r = O.gemm_tn_f64(dq(qdy, "col"), dq(qa, "col"))
    qdh = O.quantize_mxfp8(O.dgelu_bf16(da_r, qh["row"], qh["row_scale"]))
    dx_r = O.gemm_tn_f64(dq(qdh, "row"), dq(qw1, "col"))
    dw1_r = O.gemm_tn_f64(dq(qdh, "col"), dq(qx, "col"))
    for name, got, ref in (("y", y, y_r), ("dw2", dw2, dw2_r), ("dx", dx, dx_r),
                           ("dw1", dw1, dw1_r)):
        c = O.bf16_to_f32(from_dev_bf16(got)).astype(np.float64)
        err = float(np.max(np.abs(c - ref)) / np.max(np.abs(ref)))
        assert err <= 1e-2, (name, err)


def test_mlp_block_fused_small():
    _mlp_fused(256, 256, 512, seed=3)


def test_mlp_block_fused_multi_tile():
    _mlp_fused(384, 512, 1024, seed=4)


def test_full_size_fused_mlp_sampled():
    """The benchmark's fused steps at full size (tokens 8192, hidden 4096, ffn 16384): every byte
    equals the unfused GPU steps. On 384 sampled tokens (first, middle and last 128) the GEMM
    stages are checked against the oracle's fp64 sums, the GeLU stages within one bf16 ulp, and
    the quantisation of h, a and dh exactly, in the row copies and the column copies."""
    M, H, Fd = 8192, 4096, 16384
    rec = F.Recipe(kind="mxfp8")
    xb = bf16_bits_normal(M, H, seed=0, stream=0)
    w1b = bf16_bits_normal(Fd, H, seed=0, stream=1, sigma=0.02)
    w2b = bf16_bits_normal(H, Fd, seed=0, stream=3, sigma=0.02)
    dyb = bf16_bits_normal(M, H, seed=0, stream=2, sigma=1e-3)
    xq = F.quantize(rec, to_dev_bf16(xb), "activation")
    w1q = F.quantize(rec, to_dev_bf16(w1b), "weight")
    w2q = F.quantize(rec, to_dev_bf16(w2b), "weight")
    dyq = F.quantize(rec, to_dev_bf16(dyb), "grad")
    # the backward pass reads h's FP8 copy made from a seeded h, which both sides quantise
    hb = bf16_bits_normal(M, Fd, seed=0, stream=5, sigma=2.0)
    _, hs_q, _ = F.gelu_quantize(rec, to_dev_bf16(hb))
    a_q, h_q = F.linear_fwd_gelu(rec, xq, w1q)
    dh_q = F.linear_dgrad_dgelu(rec, dyq, w2q, hs_q)
    h = F.linear_fwd(rec, xq, w1q)
    a_u, h_u, a_bf16 = F.gelu_quantize(rec, h, want_a_bf16=True)
    da, _ = F.linear_bwd(rec, dyq, None, w2q, want_dw=False)
    dh_u, dh_bf16 = F.dgelu_quantize(rec, da, hs_q, want_dh_bf16=True)
    torch.cuda.synchronize()
    _same_qtensor(a_q, a_u, ("row", "row_scale", "col", "col_scale"))
    _same_qtensor(h_q, h_u, ("row", "row_scale"))
    _same_qtensor(dh_q, dh_u, ("row", "row_scale", "col", "col_scale"))

    rows = np.concatenate([np.arange(0, 128), np.arange(4160, 4288), np.arange(M - 128, M)])
    # forward: fc1's GEMM stage, GeLU stage, and the quantisation of h and a
    qx = O.quantize_mxfp8(xb[rows], want_col=False)
    qw1 = O.quantize_mxfp8(w1b, want_col=False)
    h_g, a_g = from_dev_bf16(h), from_dev_bf16(a_bf16)
    ok, err = gemm_bf16_close(h_g[rows], O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]),
                                                       O.dequant_mx(qw1["row"], qw1["row_scale"])))
    assert ok, err
    _within_one_ulp(a_g[rows], O.gelu_bf16(h_g[rows]))
    _check_copies(h_q, h_g, M, Fd, rows)
    _check_copies(a_q, a_g, M, Fd, rows)

    # backward: fc2's dgrad stage, the dGeLU stage and the quantisation of dh
    qh = O.quantize_mxfp8(hb[rows], want_col=False)
    assert np.array_equal(_np(hs_q.row)[rows], qh["row"])
    qdy = O.quantize_mxfp8(dyb[rows], want_col=False)
    qw2t = O.quantize_mxfp8(np.ascontiguousarray(w2b.T), want_col=False)
    da_g, dh_g = from_dev_bf16(da), from_dev_bf16(dh_bf16)
    ok, err = gemm_bf16_close(da_g[rows], O.gemm_tn_f64(O.dequant_mx(qdy["row"], qdy["row_scale"]),
                                                        O.dequant_mx(qw2t["row"], qw2t["row_scale"])))
    assert ok, err
    _within_one_ulp(dh_g[rows], O.dgelu_bf16(da_g[rows], qh["row"], qh["row_scale"]))
    _check_copies(dh_q, dh_g, M, Fd, rows)
