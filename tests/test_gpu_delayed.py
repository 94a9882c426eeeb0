"""GPU parity of delayed scaling over a sequence of steps: the cast uses the scale derived from
the previous steps' amax history, the fused amax is recorded, and fp8_amax_update pushes it.
Checked bit-exactly against the oracle's DelayedScaling at every step (scale, amax, codes)."""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, from_dev_bf16, gemm_bf16_close, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import STREAM_STEP0, bf16_bits_normal, sigma_schedule

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _run_sequence(M, K, steps, L, margin=0, check_codes_every=1, gemm=False, algo="max",
                  w_history=False):
    """Delayed scaling of X_t over `steps` steps. The weight W is cast once with its initial
    scale 1, or, with w_history, re-cast every step with the scale from its own amax history,
    which fp8_amax_update advances after every step as it does X's."""
    rec = F.Recipe(kind="delayed", amax_history_len=L, margin=margin, amax_compute_algo=algo)
    state = F.DelayedState(rec)
    oracle = O.DelayedScaling(L, margin, algo=algo)
    sig = sigma_schedule(steps)
    wb = bf16_bits_normal(K, K, seed=0, stream=1, sigma=0.02)
    wd = to_dev_bf16(wb)
    wstate = F.DelayedState(rec, role="weight")
    w_oracle = O.DelayedScaling(L, margin, algo=algo)
    w_amax = O.amax_of(wb)
    wq = F.quantize(rec, wd, "weight", out=wstate.bind(F.empty_qtensor(rec, K, K, "weight")))
    q = state.bind(F.empty_qtensor(rec, M, K))
    for t in range(steps):
        xb = bf16_bits_normal(M, K, seed=0, stream=STREAM_STEP0 + t, sigma=sig[t])
        if w_history and t > 0:
            F.quantize(rec, wd, "weight", out=wq)     # W's scale from its own history
        F.quantize(rec, to_dev_bf16(xb), out=q)
        if gemm:
            y = F.linear_fwd(rec, q, wq)
        used_scale = q.scale.clone()
        w_used_scale = wq.scale.clone()
        F.amax_update(rec, state, q.amax)
        if w_history:
            F.amax_update(rec, wstate, wq.amax)
        torch.cuda.synchronize()
        if t % check_codes_every == 0:
            ref = oracle.quantize(xb)
            assert np.array_equal(q.row.cpu().numpy(), ref["row"]), t
            assert np.array_equal(q.col.cpu().numpy(), ref["col"]), t
        else:
            ref = dict(amax=O.amax_of(xb), scale=oracle.scale)
        assert used_scale.cpu().numpy()[0].tobytes() == np.float32(ref["scale"]).tobytes(), t
        assert q.amax.cpu().numpy()[0].tobytes() == np.float32(ref["amax"]).tobytes(), t
        if w_history:
            assert w_used_scale.cpu().numpy()[0].tobytes() == \
                np.float32(w_oracle.scale).tobytes(), t
            assert wq.amax.cpu().numpy()[0].tobytes() == np.float32(w_amax).tobytes(), t
        if gemm and t % check_codes_every == 0:
            qw = w_oracle.quantize(wb)                 # W cast with the scale it was given
            if w_history:
                assert np.array_equal(wq.row.cpu().numpy(), qw["row"]), t
            rows = np.arange(M) if M <= 1024 else np.unique(np.concatenate(
                [np.arange(128), np.arange(M - 128, M),
                 np.random.default_rng(t).choice(M, 128, replace=False)]))
            r = O.gemm_tn_f64(O.dequant_tensor(ref["row"][rows], ref["scale_inv"]),
                              O.dequant_tensor(qw["row"], qw["scale_inv"]))
            ok, err = gemm_bf16_close(from_dev_bf16(y)[rows], r)
            assert ok, (t, err)
        oracle.update(ref["amax"])
        assert state.scale.cpu().numpy()[0].tobytes() == np.float32(oracle.scale).tobytes(), t
        assert state.scale_inv.cpu().numpy()[0].tobytes() == \
            np.float32(oracle.scale_inv).tobytes(), t
        if w_history:
            w_oracle.update(w_amax)
            assert wstate.scale.cpu().numpy()[0].tobytes() == \
                np.float32(w_oracle.scale).tobytes(), t
    assert np.array_equal(state.history.cpu().numpy(), oracle.history)
    assert int(state.head.item()) == oracle.head
    if w_history:
        assert np.array_equal(wstate.history.cpu().numpy(), w_oracle.history)
        assert int(wstate.head.item()) == w_oracle.head


def test_short_history_wraps():
    _run_sequence(256, 384, steps=12, L=4, gemm=True)


def test_weight_history_wraps():
    """W with its own delayed history: step 0 casts it with scale 1, later steps with the
    scale its recorded amax gives."""
    _run_sequence(256, 384, steps=8, L=3, gemm=True, w_history=True)


def test_most_recent_algo():
    """--fp8-amax-compute-algo most_recent: the newest amax alone sets the next scale."""
    _run_sequence(256, 384, steps=10, L=4, algo="most_recent")


def test_margin_and_long_history():
    _run_sequence(128, 256, steps=20, L=1024, margin=2)


def test_history_longer_than_block():
    # history length above the update kernel's thread count exercises the strided reduction
    _run_sequence(128, 128, steps=6, L=3000)


def test_full_size_64_steps():
    """X_t 8192 x 4096 N(0, sigma_t), sigma_t log-uniform in [0.5, 4], W 4096 x 4096 with its
    own history, history length 1024, max, margin 0, fprop each step. Scales, amaxes and both
    histories checked at all 64 steps, codes and the GEMM at every 16th."""
    _run_sequence(8192, 4096, steps=64, L=1024, check_codes_every=16, gemm=True,
                  w_history=True)
