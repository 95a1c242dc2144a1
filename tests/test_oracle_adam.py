"""Pins of the oracle's mixed-precision AdamW step: closed forms, torch, skip, clip, padding.

The optimizer state each rank keeps for its partition is the fp32 master weight, the
Adam momentum and the variance (ZeRO explainer, Chapter 02 "Memory per parameter").
"""
import numpy as np
import pytest
import torch

import oracle


def f32(x):
    return float(np.float32(x))


def rand_f16(rng, n, scale):
    return (rng.standard_normal(n) * scale).astype(np.float16).view(np.uint16)


def fresh_state(n, rng=None, master_sigma=0.0):
    master = np.zeros(n, np.float32)
    if rng is not None:
        master = (rng.standard_normal(n) * master_sigma).astype(np.float32)
    return master, np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)


def test_first_step_closed_form_without_decay():
    # m = v = 0, t' = 1, wd = 0: m_hat = g, v_hat = g^2, delta = -lr * g / (|g| + eps)
    rng = np.random.default_rng(10)
    n, ls = 20000, 1024.0
    contrib = [rand_f16(rng, n, 1e-3 * ls) for _ in range(4)]
    hp = oracle.Hyper(lr=1e-3, weight_decay=0.0)
    master, m, v, p16 = fresh_state(n)
    sc = oracle.step(contrib, master, m, v, p16, ls, 0.0, hp, 0)
    assert sc.step == 1 and sc.skipped == 0 and sc.clip_coef == 1.0
    g = oracle.reduce(contrib).astype(np.float64) * np.float64(np.float32(1.0 / ls))
    lr, eps = f32(1e-3), f32(1e-8)
    delta = -lr * g / (np.abs(g) + eps)
    assert np.allclose(master, delta, rtol=1e-6, atol=0)
    assert np.allclose(m, f32(1 - f32(0.9)) * g, rtol=1e-6, atol=0)
    assert np.allclose(v, f32(1 - f32(0.999)) * g * g, rtol=1e-6, atol=0)
    assert np.array_equal(p16, master.astype(np.float16).view(np.uint16))


def test_first_step_closed_form_with_decay():
    # with weight decay: delta = -lr*wd*p - lr * g / (|g| + eps)
    rng = np.random.default_rng(11)
    n, ls = 20000, 1024.0
    contrib = [rand_f16(rng, n, 1e-3 * ls) for _ in range(4)]
    hp = oracle.Hyper(lr=1e-3, weight_decay=0.01)
    master, m, v, p16 = fresh_state(n, rng, 0.02)
    p0 = master.astype(np.float64).copy()
    oracle.step(contrib, master, m, v, p16, ls, 0.0, hp, 0)
    g = oracle.reduce(contrib).astype(np.float64) * np.float64(np.float32(1.0 / ls))
    lr, wd, eps = f32(1e-3), f32(0.01), f32(1e-8)
    expect = p0 - lr * wd * p0 - lr * g / (np.abs(g) + eps)
    # two fp32 roundings of terms no larger than max(|p0|, |delta|): a few ulps of that
    mag = np.maximum(np.abs(p0), np.abs(expect)).astype(np.float32)
    assert np.all(np.abs(master - expect) <= 4 * np.spacing(mag))


def test_matches_torch_adamw_over_several_steps():
    rng = np.random.default_rng(12)
    n, ls, clip, steps = 5000, 4096.0, 1.0, 6
    hp = oracle.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    master, m, v, p16 = fresh_state(n, rng, 0.02)
    p = torch.nn.Parameter(torch.from_numpy(master.copy()))
    opt = torch.optim.AdamW([p], lr=f32(hp.lr), betas=(f32(hp.beta1), f32(hp.beta2)),
                            eps=f32(hp.eps), weight_decay=f32(hp.weight_decay),
                            foreach=False)
    t = 0
    for _ in range(steps):
        contrib = [rand_f16(rng, n, 1e-2 * ls) for _ in range(8)]
        gsum = oracle.reduce(contrib)
        sc = oracle.step(contrib, master, m, v, p16, ls, clip, hp, t)
        t = sc.step
        assert sc.clip_coef < 1.0  # norm ~ 2.0 with these draws: clipping is active
        p.grad = torch.from_numpy(gsum * np.float32(sc.s))
        opt.step()
        st = opt.state[p]
        # op orders differ (torch uses lerp for m and folds the bias corrections into
        # the step size), so agreement is to rounding, with a floor near cancellation
        tm, tv = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        assert np.allclose(master, p.detach().numpy(), rtol=1e-5, atol=1e-8)
        assert np.allclose(m, tm, rtol=1e-5, atol=1e-6 * np.abs(tm).max())
        assert np.allclose(v, tv, rtol=1e-5, atol=1e-6 * np.abs(tv).max())


def test_clip_coefficient_matches_torch_clip_grad_norm():
    rng = np.random.default_rng(13)
    ls = 65536.0
    for clip, scale in [(1.0, 1e-3), (1.0, 1e-5), (0.5, 1e-4), (0.0, 1e-3)]:
        contrib = [rand_f16(rng, 3000, scale * ls) for _ in range(8)]
        gsum = oracle.reduce(contrib)
        bad, ss = oracle.stats(gsum)
        sc = oracle.scalars(bad, ss, ls, clip, oracle.Hyper(), 0)
        grad = torch.from_numpy(gsum.astype(np.float64) / ls)
        q = torch.nn.Parameter(torch.zeros_like(grad))
        q.grad = grad.clone()
        if clip > 0:
            total = torch.nn.utils.clip_grad_norm_([q], max_norm=clip).item()
            assert sc.norm == pytest.approx(total, rel=1e-12)
            coef_torch = (q.grad / grad)[grad != 0].mean().item()
            assert sc.clip_coef == pytest.approx(coef_torch, rel=1e-9)
        else:
            assert sc.clip_coef == 1.0
        assert sc.s == np.float32(sc.clip_coef / ls)


def test_overflow_step_leaves_state_bit_identical():
    rng = np.random.default_rng(14)
    n = 4000
    contrib = [rand_f16(rng, n, 1.0) for _ in range(16)]
    contrib[5][1234] = 0x7C00
    master, m, v, p16 = fresh_state(n, rng, 0.02)
    m[:] = rng.standard_normal(n).astype(np.float32)
    v[:] = np.abs(rng.standard_normal(n)).astype(np.float32)
    p16[:] = rng.integers(0, 30000, n).astype(np.uint16)
    before = [a.copy() for a in (master, m, v, p16)]
    sc = oracle.step(contrib, master, m, v, p16, 4096.0, 1.0, oracle.Hyper(), 2)
    assert sc.overflow == 1 and sc.skipped == 1 and sc.step == 2
    for a, b in zip((master, m, v, p16), before):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_padding_state_is_untouched():
    rng = np.random.default_rng(15)
    n, nv = 64, 40
    contrib = [rand_f16(rng, n, 100.0) for _ in range(3)]
    for c in contrib:
        c[nv:] = 0x7E00  # NaN in padding must not count as overflow
    master, m, v, p16 = fresh_state(n)
    for _ in range(5):
        sc = oracle.step(contrib, master, m, v, p16, 128.0, 0.0, oracle.Hyper(), 0, n_valid=nv)
        assert sc.overflow == 0
    assert not master[nv:].any() and not m[nv:].any() and not v[nv:].any()
    assert not p16[nv:].any()
    assert master[:nv].any()


def test_zero_gradient_keeps_zero_state():
    n = 32
    contrib = [np.zeros(n, np.uint16) for _ in range(4)]
    master, m, v, p16 = fresh_state(n)
    for t in range(3):
        sc = oracle.step(contrib, master, m, v, p16, 1.0, 1.0, oracle.Hyper(), t)
        assert sc.norm == 0.0 and sc.clip_coef == 1.0 and sc.step == t + 1
    assert not master.any() and not m.any() and not v.any() and not p16.any()


def test_bias_correction_scalars():
    hp = oracle.Hyper(beta1=0.9, beta2=0.999)
    for t in [0, 1, 9, 99, 10**6]:
        sc = oracle.scalars(0, 0, 1.0, 0.0, hp, t)
        tp = t + 1
        assert sc.bc1 == np.float32(1 - np.float64(np.float32(0.9)) ** tp)
        assert sc.bc2 == np.float32(1 - np.float64(np.float32(0.999)) ** tp)
        assert sc.decay == np.float32(1 - np.float64(np.float32(1e-3)) * np.float64(np.float32(0.01)))


def test_param16_is_rounded_master():
    rng = np.random.default_rng(16)
    n = 10000
    contrib = [rand_f16(rng, n, 1e3) for _ in range(2)]
    master, m, v, p16 = fresh_state(n, rng, 3.0)
    oracle.step(contrib, master, m, v, p16, 1.0, 0.0, oracle.Hyper(lr=0.1), 0)
    assert np.array_equal(p16, master.astype(np.float16).view(np.uint16))


def test_decay_is_applied_before_the_adam_term():
    # with lr * wd large, decaying after the Adam term instead of before moves the
    # result by lr^2 * wd * u, far beyond rounding: torch's AdamW decays first
    rng = np.random.default_rng(17)
    n, ls = 4000, 1.0
    hp = oracle.Hyper(lr=0.1, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.5)
    master, m, v, p16 = fresh_state(n, rng, 1.0)
    p = torch.nn.Parameter(torch.from_numpy(master.copy()))
    opt = torch.optim.AdamW([p], lr=f32(hp.lr), betas=(f32(hp.beta1), f32(hp.beta2)),
                            eps=f32(hp.eps), weight_decay=f32(hp.weight_decay), foreach=False)
    t = 0
    for _ in range(3):
        contrib = [rand_f16(rng, n, 1.0) for _ in range(2)]
        gsum = oracle.reduce(contrib)
        sc = oracle.step(contrib, master, m, v, p16, ls, 0.0, hp, t)
        t = sc.step
        p.grad = torch.from_numpy(gsum * np.float32(sc.s))
        opt.step()
        assert np.allclose(master, p.detach().numpy(), rtol=1e-5, atol=1e-6)
    # the other order would be off by about lr^2 * wd = 5e-3 per step
    assert np.abs(master - p.detach().numpy()).max() < 1e-4
