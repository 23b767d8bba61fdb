"""Weights stored in NVFP4 and updated in place ("fp4-train", Correctness and
the Usage loop): with sub-step updates round-to-nearest never leaves its
starting loss, while stochastic rounding and error feedback keep descending,
error feedback further, and fp32 further still.

Two synthetic toys, the page's two (its own data and models are not given):
a linear regression, targets Y = X W*^T, and a small MLP (tanh hidden layer)
fitting a teacher MLP.  Each weight lives only as qdq(W - lr * grad) (the value
the tensor cores use), with the step size chosen so one update is a small
fraction of a quantization step.  The CPU tests run the oracle's qdq (a pin of
its SR / EF behaviour against the page's claim: RTN stuck, SR and EF near the
full-precision loss, EF the closer); the GPU tests run the library's and
require its loss curves to equal the oracle's bit for bit.
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


def _oracle_qdq(rounding, ef, shape=(16, 128), seed=7):
    res = np.zeros(shape, np.float32) if ef else None

    def f(W, t):
        o = oracle.qdq(W, rounding=rounding, residual=res, seed=seed, step=t)
        return (o["out"].astype(np.uint32) << 16).view(np.float32)      # bf16 bits -> fp32
    return f


# ---- the small MLP: X [512,64] -> tanh(X W1^T) [512,64] -> W2 [8,64] ---------------------
MLP_STEPS, MLP_LR = 300, 0.05
MLP_SHAPES = ((64, 64), (8, 64))


def _mlp_problem():
    rng = np.random.default_rng(77)
    X = rng.standard_normal((512, 64)).astype(np.float32)
    A1 = (rng.standard_normal(MLP_SHAPES[0]) * 0.3).astype(np.float32)
    A2 = (rng.standard_normal(MLP_SHAPES[1]) * 0.3).astype(np.float32)
    Y = (np.tanh(X @ A1.T) @ A2.T).astype(np.float32)
    W1 = (A1 + rng.standard_normal(A1.shape).astype(np.float32) * 0.3).astype(np.float32)
    W2 = (A2 + rng.standard_normal(A2.shape).astype(np.float32) * 0.3).astype(np.float32)
    return X, Y, W1, W2


def _train_mlp(q1, q2):
    """q1, q2: the stored-weight maps of the two layers; returns the loss curve."""
    X, Y, W1, W2 = _mlp_problem()
    W1, W2 = q1(W1, 0), q2(W2, 0)
    losses = []
    for t in range(MLP_STEPS):
        H = np.tanh(X @ W1.T)
        R = H @ W2.T - Y
        losses.append(float((R ** 2).mean()))
        G2 = (R.T @ H) / X.shape[0]
        G1 = (((R @ W2) * (1 - H ** 2)).T @ X) / X.shape[0]
        W1 = q1((W1 - np.float32(MLP_LR) * G1).astype(np.float32), t + 1)
        W2 = q2((W2 - np.float32(MLP_LR) * G2).astype(np.float32), t + 1)
    return np.array(losses)


def _check_mlp(curves):
    rtn, sr, ef, f32 = curves["rtn"], curves["sr"], curves["ef"], curves["fp32"]
    half = MLP_STEPS // 2
    assert rtn[-1] == rtn[half] and rtn[-1] > 0.8 * rtn[0]   # round-to-nearest stops moving, high
    assert sr[-1] < 0.1 * sr[0] and ef[-1] < 0.1 * ef[0]     # SR and EF keep descending
    assert ef[-1] < sr[-1]                                   # EF ends closer to full precision
    assert f32[-1] < ef[-1] < 2 * f32[-1]                    # ... within a factor 2 of it
    assert rtn[-1] > 10 * sr[-1]


def _oracle_mlp_curves():
    out = {}
    for name, rnd, ef in (("rtn", oracle.RTN, False), ("sr", oracle.SR, False), ("ef", oracle.RTN, True)):
        out[name] = _train_mlp(_oracle_qdq(rnd, ef, MLP_SHAPES[0], 11), _oracle_qdq(rnd, ef, MLP_SHAPES[1], 12))
    out["fp32"] = _train_mlp(lambda W, t: W, lambda W, t: W)
    return out


def test_stored_weight_mlp_oracle():
    _check_mlp(_oracle_mlp_curves())


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


@pytest.mark.gpu
def test_stored_weight_mlp_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_block_quantization_quantize_gb300 as nv
    nv.build()
    nv.load_library()

    def lib_qdq(rounding, ef, shape, seed):
        res = torch.zeros(shape, dtype=torch.float32, device="cuda") if ef else None

        def f(W, t):
            o = nv.nvfp4_qdq(torch.from_numpy(W).cuda(), rounding=rounding, residual=res, seed=seed, step=t)
            return o["out"].float().cpu().numpy()
        return f

    curves = {}
    for name, rnd, ef in (("rtn", "rtn", False), ("sr", "sr", False), ("ef", "rtn", True)):
        curves[name] = _train_mlp(lib_qdq(rnd, ef, MLP_SHAPES[0], 11), lib_qdq(rnd, ef, MLP_SHAPES[1], 12))
    curves["fp32"] = _train_mlp(lambda W, t: W, lambda W, t: W)
    _check_mlp(curves)
    ref = _oracle_mlp_curves()
    for k in ("rtn", "sr", "ef"):
        assert np.array_equal(curves[k], ref[k]), k


@pytest.mark.gpu
@pytest.mark.parametrize("stochastic", [False, True])
def test_error_feedback_state_runs_the_usage_loop(stochastic):
    """The page's stored-weight loop through ErrorFeedback (W = ef.qdq(name,
    W - lr * grad, step)): its residual is carried across the steps, and the
    loss curve equals the oracle's with the same residual, bit for bit."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_block_quantization_quantize_gb300 as nv
    from nvfp4_block_quantization_quantize_gb300.error_feedback import ErrorFeedback
    nv.build()
    nv.load_library()
    ef = ErrorFeedback(stochastic=stochastic, seed=7)
    curve = _train(lambda W, t: ef.qdq("layer0.weight", torch.from_numpy(W).cuda(), step=t).float().cpu().numpy())
    assert ef.names() == ["layer0.weight"]
    ref = _train(_oracle_qdq(oracle.SR if stochastic else oracle.RTN, True))
    assert np.array_equal(curve, ref)
