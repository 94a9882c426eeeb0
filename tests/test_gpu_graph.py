"""The library launches only on the caller's stream, never allocates and never synchronises,
so whole steps can be captured in a CUDA graph. A captured MXFP8 MLP step (grouped quantize of
X, W1 and W2, fused epilogues) and a delayed-scaling step (quantize, fprop, history update)
replayed from the graph must give the same bytes as the same calls run eagerly."""
import pytest
import torch

from helpers import cuda_ok, to_dev_bf16
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _capture_and_compare(step, outputs):
    step()                                           # eager run (also sets kernel attributes)
    torch.cuda.synchronize()
    ref = [t.clone() for t in outputs]
    for t in outputs:
        t.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t in outputs:
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outputs, ref):
        assert torch.equal(a, b)


def test_graph_mxfp8_mlp_step():
    rec = F.Recipe(kind="mxfp8")
    M, H, Fd = 256, 256, 512
    x = to_dev_bf16(bf16_bits_normal(M, H, seed=1, stream=0))
    w1 = to_dev_bf16(bf16_bits_normal(Fd, H, seed=1, stream=1, sigma=0.02))
    w2 = to_dev_bf16(bf16_bits_normal(H, Fd, seed=1, stream=3, sigma=0.02))
    dy = to_dev_bf16(bf16_bits_normal(M, H, seed=1, stream=2, sigma=1e-3))
    e = F.empty_qtensor
    xq, w1q, w2q, dyq = (e(rec, M, H, "activation"), e(rec, Fd, H, "weight"),
                         e(rec, H, Fd, "weight"), e(rec, M, H, "grad"))
    aq, hq, dhq = (e(rec, M, Fd, "activation"), e(rec, M, Fd, "activation", want_col=False),
                   e(rec, M, Fd, "grad"))
    y, dx = torch.empty_like(x), torch.empty_like(x)
    dw1, dw2 = torch.empty_like(w1), torch.empty_like(w2)

    def step():
        # X, W1 and W2 in one grouped launch, as the benchmark step does
        F.quantize_group(rec, [x, w1, w2], ["activation", "weight", "weight"],
                         outs=[xq, w1q, w2q])
        F.linear_fwd_gelu(rec, xq, w1q, a_q=aq, h_q=hq)
        F.linear_fwd(rec, aq, w2q, y=y)
        F.quantize(rec, dy, "grad", out=dyq)
        F.linear_dgrad_dgelu(rec, dyq, w2q, hq, dh_q=dhq)
        F.linear_bwd(rec, dyq, aq, None, want_dx=False, dw=dw2)
        F.linear_bwd(rec, dhq, xq, w1q, dx=dx, dw=dw1)

    _capture_and_compare(step, [y, dx, dw1, dw2, aq.row, aq.col, dhq.row, dhq.col, xq.row,
                                xq.col, w1q.col, w2q.row])


def test_graph_delayed_step_with_history():
    rec = F.Recipe(kind="delayed", amax_history_len=8)
    M, K, N = 256, 384, 256
    x = to_dev_bf16(bf16_bits_normal(M, K, seed=2, stream=0))
    w = to_dev_bf16(bf16_bits_normal(N, K, seed=2, stream=1, sigma=0.02))
    sx, sw = F.DelayedState(rec), F.DelayedState(rec, role="weight")
    xq = sx.bind(F.empty_qtensor(rec, M, K, "activation"))
    wq = sw.bind(F.empty_qtensor(rec, N, K, "weight"))
    ws = torch.empty(max(1, F.workspace_bytes(rec, M, K)), dtype=torch.uint8, device="cuda")
    wsw = torch.empty(max(1, F.workspace_bytes(rec, N, K)), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    snapshot = [t.clone() for t in (sx.history, sx.head, sx.scale, sx.scale_inv,
                                    sw.history, sw.head, sw.scale, sw.scale_inv)]

    def restore():
        for t, v in zip((sx.history, sx.head, sx.scale, sx.scale_inv,
                         sw.history, sw.head, sw.scale, sw.scale_inv), snapshot):
            t.copy_(v)

    def step():
        restore()                                    # every run starts from the same history
        F.quantize(rec, x, "activation", out=xq, workspace=ws)
        F.quantize(rec, w, "weight", out=wq, workspace=wsw)
        F.linear_fwd(rec, xq, wq, y=y)
        F.amax_update(rec, sx, xq.amax)
        F.amax_update(rec, sw, wq.amax)

    _capture_and_compare(step, [y, xq.row, xq.col, sx.history, sx.scale, sw.scale])
