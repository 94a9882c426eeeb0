"""GPU parity of the fused MLP steps (MXFP8): fc1 with the GeLU step in the GEMM epilogue
(h's FP8 row copy plus a = gelu(h) as row and column copies, h never stored in bf16), and the
dgrad of fc2 with the GeLU backward in the epilogue (dh = da * gelu'(h) as row and column
copies, da never stored).

Each fused output is checked two ways:
- against the oracle on the same seeded inputs. The oracle's fp64 GEMM rounds to bf16 and may
  differ from the GPU's fp32 accumulation by one unit in the last place, so a 1x32 block whose
  bf16 quantiser input agrees exactly with the oracle's must agree byte for byte (codes and
  E8M0 scale); other blocks must dequantise within two E4M3 steps of the oracle's;
- against the unfused GPU steps (GEMM storing bf16, then the standalone GeLU kernel): both round
  the same fp32 accumulator to bf16 and apply the same fp32 GeLU, so every byte must agree.
"""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, from_dev_bf16, mx_untile, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _np(t):
    return t.cpu().numpy()


def _check_mx_blocks(codes, scale_plain, gpu_in, ref_in):
    """codes [R][C] and plain E8M0 scales [R][C/32] produced on the GPU from the bf16 input
    gpu_in; the oracle quantises ref_in. Returns the fraction of bit-identical blocks."""
    R, C = ref_in.shape
    ref = O.quantize_mxfp8(ref_in, want_col=False)
    same = (gpu_in == ref_in).reshape(R, C // 32, 32).all(axis=2)
    got = codes.reshape(R, C // 32, 32)
    rc = ref["row"].reshape(R, C // 32, 32)
    assert np.array_equal(got[same], rc[same])
    assert np.array_equal(scale_plain[same], ref["row_scale"][same])
    sr = O.e8m0_decode(ref["row_scale"])[:, :, None]
    dg = O.e4m3_decode(got) * O.e8m0_decode(scale_plain)[:, :, None]
    dr = O.e4m3_decode(rc) * sr
    tol = 0.25 * np.abs(dr) + 2.0 ** -9 * sr
    assert np.all((np.abs(dg - dr) <= tol)[~same])
    return float(same.mean())


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


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 256, 256), (384, 512, 256),
                                   (512, 384, 512), (256, 128, 384)])
def test_fc1_gelu_fused(M, N, K):
    rec, xb, wb, xq, wq = _fc1(M, N, K, seed=M + N)
    a_q, h_q = F.linear_fwd_gelu(rec, xq, wq)
    # unfused GPU steps
    h = F.linear_fwd(rec, xq, wq)
    a_u, h_u, a_bf16 = F.gelu_quantize(rec, h, want_a_bf16=True)
    torch.cuda.synchronize()
    _same_qtensor(a_q, a_u, ("row", "row_scale", "col", "col_scale"))
    _same_qtensor(h_q, h_u, ("row", "row_scale"))
    # oracle
    qx, qw = O.quantize_mxfp8(xb, want_col=False), O.quantize_mxfp8(wb, want_col=False)
    h_r = O.f64_to_bf16(O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]),
                                      O.dequant_mx(qw["row"], qw["row_scale"])))
    a_r = O.gelu_bf16(h_r)
    h_g, a_g = from_dev_bf16(h), from_dev_bf16(a_bf16)
    f = _check_mx_blocks(_np(h_q.row), mx_untile(_np(h_q.row_scale), M, N), h_g, h_r)
    assert f > 0.5
    _check_mx_blocks(_np(a_q.row), mx_untile(_np(a_q.row_scale), M, N), a_g, a_r)
    _check_mx_blocks(_np(a_q.col), mx_untile(_np(a_q.col_scale), N, M),
                     np.ascontiguousarray(a_g.T), np.ascontiguousarray(a_r.T))


@pytest.mark.parametrize("M,Fd,H", [(128, 256, 128), (256, 256, 256), (384, 512, 256),
                                    (512, 384, 128)])
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
    # oracle: da = dY . (W2^T)^T from the column copy of W2, then gelu' of the FP8 h
    qh = O.quantize_mxfp8(hb, want_col=False)
    assert np.array_equal(_np(h_q.row), qh["row"])
    qdy = O.quantize_mxfp8(dyb, want_col=False)
    qw2t = O.quantize_mxfp8(np.ascontiguousarray(w2b.T), want_col=False)
    da_r = O.f64_to_bf16(O.gemm_tn_f64(O.dequant_mx(qdy["row"], qdy["row_scale"]),
                                       O.dequant_mx(qw2t["row"], qw2t["row_scale"])))
    dh_r = O.dgelu_bf16(da_r, qh["row"], qh["row_scale"])
    dh_g = from_dev_bf16(dh_bf16)
    _check_mx_blocks(_np(dh_q.row), mx_untile(_np(dh_q.row_scale), M, Fd), dh_g, dh_r)
    _check_mx_blocks(_np(dh_q.col), mx_untile(_np(dh_q.col_scale), Fd, M),
                     np.ascontiguousarray(dh_g.T), np.ascontiguousarray(dh_r.T))


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
    da_r = O.f64_to_bf16(O.gemm_tn_f64(O.dequant_mx(qdy["row"], qdy["row_scale"]),
                                       O.dequant_mx(qw2t["row"], qw2t["row_scale"])))
    dh_r = O.dgelu_bf16(da_r, qh["row"], qh["row_scale"])
    dh_g = from_dev_bf16(dh_bf16)
    # NaN blocks of dh (from the Inf / NaN h blocks): codes and scale marked NaN on both sides
    nan_r = np.isnan(O.bf16_to_f32(dh_r)).reshape(M, Fd // 32, 32).any(axis=2)
    assert np.array_equal(nan_r, (mx_untile(_np(dh_q.row_scale), M, Fd) == 255))
    fin_rows = ~nan_r.any(axis=1)
    _check_mx_blocks(_np(dh_q.row)[fin_rows], mx_untile(_np(dh_q.row_scale), M, Fd)[fin_rows],
                     dh_g[fin_rows], dh_r[fin_rows])


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
    equals the unfused GPU steps, and three 32-row blocks of tokens (first, middle, last) are
    checked against the oracle in both the row copies and the column copies."""
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

    blocks = [0, 131, M // 32 - 1]
    rows = np.concatenate([np.arange(32 * b, 32 * b + 32) for b in blocks])
    qx = O.quantize_mxfp8(xb[rows], want_col=False)
    qw1 = O.quantize_mxfp8(w1b, want_col=False)
    h_r = O.f64_to_bf16(O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]),
                                      O.dequant_mx(qw1["row"], qw1["row_scale"])))
    a_r = O.gelu_bf16(h_r)
    h_g, a_g = from_dev_bf16(h)[rows], from_dev_bf16(a_bf16)[rows]
    hs = mx_untile(_np(h_q.row_scale), M, Fd)[rows]
    assert _check_mx_blocks(_np(h_q.row)[rows], hs, h_g, h_r) > 0.5
    _check_mx_blocks(_np(a_q.row)[rows], mx_untile(_np(a_q.row_scale), M, Fd)[rows], a_g, a_r)
    a_col, a_cs = _np(a_q.col), mx_untile(_np(a_q.col_scale), Fd, M)
    for i, b in enumerate(blocks):
        sl = slice(32 * i, 32 * i + 32)
        _check_mx_blocks(np.ascontiguousarray(a_col[:, 32 * b:32 * b + 32]), a_cs[:, b:b + 1],
                         np.ascontiguousarray(a_g[sl].T), np.ascontiguousarray(a_r[sl].T))

    # backward
    qh = O.quantize_mxfp8(hb[rows], want_col=False)
    assert np.array_equal(_np(hs_q.row)[rows], qh["row"])
    qdy = O.quantize_mxfp8(dyb[rows], want_col=False)
    qw2t = O.quantize_mxfp8(np.ascontiguousarray(w2b.T), want_col=False)
    da_r = O.f64_to_bf16(O.gemm_tn_f64(O.dequant_mx(qdy["row"], qdy["row_scale"]),
                                       O.dequant_mx(qw2t["row"], qw2t["row_scale"])))
    dh_r = O.dgelu_bf16(da_r, qh["row"], qh["row_scale"])
    dh_g = from_dev_bf16(dh_bf16)[rows]
    _check_mx_blocks(_np(dh_q.row)[rows], mx_untile(_np(dh_q.row_scale), M, Fd)[rows], dh_g,
                     dh_r)
    d_col, d_cs = _np(dh_q.col), mx_untile(_np(dh_q.col_scale), Fd, M)
    for i, b in enumerate(blocks):
        sl = slice(32 * i, 32 * i + 32)
        _check_mx_blocks(np.ascontiguousarray(d_col[:, 32 * b:32 * b + 32]), d_cs[:, b:b + 1],
                         np.ascontiguousarray(dh_g[sl].T), np.ascontiguousarray(dh_r[sl].T))
