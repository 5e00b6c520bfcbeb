"""Pins of the oracle's encoder against closed forms, invariants, brute force and an
independent restatement with torch CPU ops (torch.nn.functional).

Sources: "whisper 0.9.0 API", model.nu (conv1 k=3 s=1 pad=1, conv2 k=3 s=2 pad=1,
3000 -> 1500 frames, stored positions, N x [LN -> non-causal self-attn -> +res,
LN -> fc1 -> GELU -> fc2 -> +res], final LN; k_proj has no bias) and kernels.nu
(LayerNorm with bias, erf GELU, attention scores q.k / sqrt(hd) with no causal mask).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import whisper_ref as R
from whisper_audio_encoder_gb300 import synth

RNG = np.random.default_rng(99)


# ---------------------------------------------------------------- GELU
def test_gelu_closed_values():
    # GELU(x) = x Phi(x); Phi(1) = 0.841344746068543, Phi(-1) = 1 - Phi(1)
    assert R.gelu(np.array(0.0)) == 0.0
    assert R.gelu(np.array(1.0)) == pytest.approx(0.8413447460685429, abs=1e-15)
    assert R.gelu(np.array(-1.0)) == pytest.approx(-0.15865525393145707, abs=1e-15)
    assert R.gelu(np.array(2.0)) == pytest.approx(2 * 0.9772498680518208, abs=1e-15)


def test_gelu_is_erf_form_not_tanh():
    x = np.linspace(-6, 6, 2001)
    ref = F.gelu(torch.from_numpy(x), approximate="none").numpy()
    tanh = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.max(np.abs(R.gelu(x) - ref)) < 1e-12
    assert np.max(np.abs(R.gelu(x) - tanh)) > 1e-4            # the two forms are distinguishable


# ---------------------------------------------------------------- LayerNorm
def test_layer_norm_vs_torch_and_invariants():
    x = RNG.standard_normal((50, 384)) * 3 + 1.5
    g = 1 + 0.3 * RNG.standard_normal(384)
    b = 0.2 * RNG.standard_normal(384)
    y = R.layer_norm(x, g, b)
    ref = F.layer_norm(torch.from_numpy(x), (384,), torch.from_numpy(g), torch.from_numpy(b), eps=1e-5)
    assert np.max(np.abs(y - ref.numpy())) < 1e-12
    y1 = R.layer_norm(x, np.ones(384), np.zeros(384))
    assert np.allclose(y1.mean(axis=1), 0, atol=1e-12)
    assert np.allclose(y1.var(axis=1), 1, atol=1e-5)           # var/(var+eps), var ~ 9


# ---------------------------------------------------------------- conv stem
def _conv_brute(x, w, b, stride):
    t_in, c_in = x.shape
    c_out = w.shape[0]
    t_out = (t_in + 2 - 3) // stride + 1
    y = np.zeros((t_out, c_out))
    for t in range(t_out):
        for o in range(c_out):
            acc = b[o]
            for j in range(3):
                s = stride * t + j - 1
                if 0 <= s < t_in:
                    for i in range(c_in):
                        acc += w[o, i, j] * x[s, i]
            y[t, o] = acc
    return y


@pytest.mark.parametrize("stride", [1, 2])
def test_conv1d_brute_force(stride):
    x = RNG.standard_normal((9, 5))
    w = RNG.standard_normal((4, 5, 3))
    b = RNG.standard_normal(4)
    assert np.max(np.abs(R.conv1d_k3(x, w, b, stride) - _conv_brute(x, w, b, stride))) < 1e-12


@pytest.mark.parametrize("stride", [1, 2])
def test_conv1d_vs_torch_and_3000_to_1500(stride):
    x = RNG.standard_normal((3000, 16))
    w = RNG.standard_normal((24, 16, 3))
    b = RNG.standard_normal(24)
    y = R.conv1d_k3(x, w, b, stride)
    ref = F.conv1d(torch.from_numpy(x.T[None]), torch.from_numpy(w), torch.from_numpy(b),
                   stride=stride, padding=1)[0].T.numpy()
    assert y.shape == ((3000, 24) if stride == 1 else (1500, 24))
    assert np.max(np.abs(y - ref)) < 1e-11


def test_stride2_output_reads_inputs_2t_minus_1_to_2t_plus_1():
    w = np.ones((1, 1, 3))
    for s, expect in ((100, {50}), (101, {50, 51}), (0, {0}), (2999, {1499})):
        x = np.zeros((3000, 1))
        x[s, 0] = 1.0
        y = R.conv1d_k3(x, w, np.zeros(1), 2)[:, 0]
        assert set(np.nonzero(y)[0].tolist()) == expect       # t with s in {2t-1, 2t, 2t+1}


# ---------------------------------------------------------------- attention
def _sdpa(q, k, v, n_head):
    t, d = q.shape
    hd = d // n_head
    split = lambda a: torch.from_numpy(a).reshape(t, n_head, hd).transpose(0, 1)[None]
    o = F.scaled_dot_product_attention(split(q), split(k), split(v), is_causal=False)
    return o[0].transpose(0, 1).reshape(t, d).numpy()


def test_attention_vs_torch_sdpa_peaked():
    q, k, v = (RNG.standard_normal((300, 128)) for _ in range(3))   # N(0,1): peaked softmax
    assert np.max(np.abs(R.attention(q, k, v, 2) - _sdpa(q, k, v, 2))) < 1e-12


def test_attention_rows_sum_to_one_and_non_causal():
    q, k, v = (RNG.standard_normal((200, 64)) for _ in range(3))
    out, probs = R.attention(q, k, v, 1, return_probs=True)
    assert np.allclose(probs[0].sum(axis=1), 1.0, atol=1e-12)
    assert np.all(probs[0][0, 1:] > 0)                 # query 0 attends to future keys
    v2 = v.copy()
    v2[-1] += 10.0                                     # perturb the last frame
    assert np.max(np.abs(R.attention(q, k, v2, 1)[0] - out[0])) > 1e-6


def test_attention_equal_keys_give_mean_of_v():
    q = RNG.standard_normal((10, 64))
    k = np.tile(RNG.standard_normal((1, 64)), (50, 1))
    v = RNG.standard_normal((50, 64))
    assert np.allclose(R.attention(q, k, v, 1), np.tile(v.mean(axis=0), (10, 1)), atol=1e-12)


def test_attention_scale_is_one_over_sqrt_64():
    q = RNG.standard_normal((2, 64))
    k = RNG.standard_normal((2, 64))
    v = np.eye(2, 64)
    _, probs = R.attention(q, k, v, 1, return_probs=True)
    s = q @ k.T / 8.0
    p = np.exp(s) / np.exp(s).sum(axis=1, keepdims=True)
    assert np.allclose(probs[0], p, atol=1e-14)


def test_k_bias_cannot_change_the_block_output():
    # softmax is invariant to adding q . b_k to a row, so whisper's missing k bias is
    # harmless to leave out, and adding one must not change the result.
    w = synth.random_weights(80, 128, 1, 512, seed=5)
    x = RNG.standard_normal((1500, 128)) * 0.5
    y0 = R.encoder_block(x, w["layers"][0], 2)
    y1 = R.encoder_block(x, w["layers"][0], 2, bk=RNG.standard_normal(128))
    assert np.max(np.abs(y0 - y1)) < 1e-9


# ---------------------------------------------------------------- full encoder
def _torch_encoder(mel, w, n_head):
    """An independent restatement of the encoder with torch.nn.functional, float64."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    x = t(mel).T[None]                                                # [1][M][3000]
    x = F.gelu(F.conv1d(x, t(w["conv1_w"]), t(w["conv1_b"]), stride=1, padding=1))
    x = F.gelu(F.conv1d(x, t(w["conv2_w"]), t(w["conv2_b"]), stride=2, padding=1))
    x = x[0].T + t(w["pos"])                                          # [1500][d]
    d = x.shape[1]
    hd = d // n_head
    heads = lambda a: a.reshape(-1, n_head, hd).transpose(0, 1)[None]
    for lw in w["layers"]:
        h = F.layer_norm(x, (d,), t(lw["ln1_g"]), t(lw["ln1_b"]), eps=1e-5)
        q = F.linear(h, t(lw["wq"]), t(lw["bq"]))
        k = F.linear(h, t(lw["wk"]))
        v = F.linear(h, t(lw["wv"]), t(lw["bv"]))
        a = F.scaled_dot_product_attention(heads(q), heads(k), heads(v))[0].transpose(0, 1).reshape(-1, d)
        x = x + F.linear(a, t(lw["wo"]), t(lw["bo"]))
        h = F.layer_norm(x, (d,), t(lw["ln2_g"]), t(lw["ln2_b"]), eps=1e-5)
        x = x + F.linear(F.gelu(F.linear(h, t(lw["w1"]), t(lw["b1"]))), t(lw["w2"]), t(lw["b2"]))
    return F.layer_norm(x, (d,), t(w["lnf_g"]), t(w["lnf_b"]), eps=1e-5).numpy()


def test_full_encoder_matches_torch_restatement():
    w = synth.random_weights(80, 128, 2, 512, seed=11, ln_random=True)
    mel = RNG.uniform(-1.0, 1.0, (3000, 80))
    y = R.encoder(mel, w, 2)
    assert y.shape == (1500, 128)
    assert np.max(np.abs(y - _torch_encoder(mel, w, 2))) < 1e-9


def test_full_window_shapes_480000_to_1500():
    w = synth.random_weights(128, 128, 1, 512, seed=3)
    mel, y = R.encode_window(np.zeros(1000, np.float32), w, 128, 2)
    assert mel.shape == (3000, 128) and y.shape == (1500, 128)


# ---------------------------------------------------------------- planted mistakes
def test_planted_mistakes_are_caught(monkeypatch):
    """Each plausible slip in the oracle must break one of the pins above."""
    x = np.linspace(-6, 6, 101)
    good = F.gelu(torch.from_numpy(x)).numpy()
    tanh_gelu = lambda a: 0.5 * a * (1 + np.tanh(math.sqrt(2 / math.pi) * (a + 0.044715 * a ** 3)))
    assert np.max(np.abs(tanh_gelu(x) - good)) > 1e-6

    # a symmetric Hann window fails the torch.hann_window comparison
    n = np.arange(400)
    sym = 0.5 - 0.5 * np.cos(2 * np.pi * n / 399)
    assert np.max(np.abs(sym - torch.hann_window(400, periodic=True, dtype=torch.float64).numpy())) > 1e-4

    # a causal mask fails the sdpa comparison
    q, k, v = (RNG.standard_normal((64, 64)) for _ in range(3))
    s = q @ k.T / 8
    s = np.where(np.tri(64) > 0, s, -np.inf)
    p = np.exp(s - s.max(1, keepdims=True))
    causal = (p / p.sum(1, keepdims=True)) @ v
    assert np.max(np.abs(causal - _sdpa(q, k, v, 1))) > 1e-3

    # a dropped positional add or a transposed conv weight breaks the full-encoder restatement
    w = synth.random_weights(80, 128, 1, 512, seed=12)
    mel = RNG.uniform(-1.0, 1.0, (3000, 80))
    ref = _torch_encoder(mel, w, 2)
    orig_stem = R.encoder_stem
    monkeypatch.setattr(R, "encoder_stem", lambda m, ww: orig_stem(m, ww) - ww["pos"])
    assert np.max(np.abs(R.encoder(mel, w, 2) - ref)) > 1e-3
    monkeypatch.setattr(R, "encoder_stem", orig_stem)
    w_t = dict(w, conv1_w=w["conv1_w"][:, :, ::-1].copy())           # taps reversed
    assert np.max(np.abs(R.encoder(mel, w_t, 2) - ref)) > 1e-3
