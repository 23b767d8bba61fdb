"""Weights stored in NVFP4 and updated in place ("fp4-train", Correctness and
the Usage loop): with sub-step updates round-to-nearest never leaves its
starting loss, while stochastic rounding and error feedback keep descending,
error feedback further, and fp32 further still.

A synthetic linear-regression toy: targets Y = X W*^T; the weight W lives only
as qdq(W - lr * grad) (the value the tensor cores use), with the step size
chosen so one update is a small fraction of a quantization step.  The CPU test
runs the oracle's qdq (a pin of its SR / EF behaviour against the page's
claim); the GPU test runs the library's.
"""
import numpy as np
import pytest

import oracle

STEPS, LR = 300, 0.02


def _problem():
    rng = np.random.default_rng(2024)
    X = rng.standard_normal((512, 128)).astype(np.float32)
    W_true = (rng.standard_normal((16, 128)) * 0.5).astype(np.float32)
    W0 = (W_true + rng.standard_normal(W_true.shape).astype(np.float32) * 0.5).astype(np.float32)
    return X, X @ W_true.T, W0


def _train(qdq):
    """qdq(W, t) -> the stored weight (fp32 array) after quantizing W at step t;
    returns the loss curve."""
    X, Y, W0 = _problem()
    W = qdq(W0, 0)
    losses = []
    for t in range(STEPS):
        R = X @ W.T - Y
        losses.append(float((R ** 2).mean()))
        G = (R.T @ X) / X.shape[0]
        W = qdq((W - np.float32(LR) * G).astype(np.float32), t + 1)
    return np.array(losses)


def _oracle_qdq(rounding, ef):
    res = np.zeros((16, 128), np.float32) if ef else None

    def f(W, t):
        o = oracle.qdq(W, rounding=rounding, residual=res, seed=7, step=t)
        return (o["out"].astype(np.uint32) << 16).view(np.float32)      # bf16 bits -> fp32
    return f


def _check(curves):
    rtn, sr, ef, f32 = curves["rtn"], curves["sr"], curves["ef"], curves["fp32"]
    assert rtn[-1] >= 0.98 * rtn[0]                  # round-to-nearest stalls
    assert sr[-1] < 0.6 * sr[0]                      # stochastic rounding descends
    assert ef[-1] < 0.6 * ef[0]                      # error feedback descends
    assert ef[-1] < sr[-1]                           # ... further than SR
    assert f32[-1] < min(sr[-1], ef[-1])             # fp32 is the reference


def test_stored_weight_toy_oracle():
    curves = {"rtn": _train(_oracle_qdq(oracle.RTN, False)),
              "sr": _train(_oracle_qdq(oracle.SR, False)),
              "ef": _train(_oracle_qdq(oracle.RTN, True)),
              "fp32": _train(lambda W, t: W)}
    _check(curves)


@pytest.mark.gpu
def test_stored_weight_toy_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_block_quantization_quantize_gb300 as nv
    nv.build()
    nv.load_library()

    def lib_qdq(rounding, ef):
        res = torch.zeros((16, 128), dtype=torch.float32, device="cuda") if ef else None

        def f(W, t):
            o = nv.nvfp4_qdq(torch.from_numpy(W).cuda(), rounding=rounding, residual=res, seed=7, step=t)
            return o["out"].float().cpu().numpy()
        return f

    curves = {"rtn": _train(lib_qdq("rtn", False)), "sr": _train(lib_qdq("sr", False)),
              "ef": _train(lib_qdq("rtn", True)), "fp32": _train(lambda W, t: W)}
    _check(curves)
    # the library's stored weights follow the oracle's exactly, so do the curves
    ref = {"sr": _train(_oracle_qdq(oracle.SR, False)), "ef": _train(_oracle_qdq(oracle.RTN, True))}
    for k in ref:
        assert np.array_equal(curves[k], ref[k]), k
