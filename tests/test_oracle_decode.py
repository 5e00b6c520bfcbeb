"""Pins of the oracle's decode step against facts fixed outside the oracle itself.

One decoder step ("whisper 0.9.0 API", model.nu, wh_decode_step: token tok at position pos,
everything before it already in the KV cache, one query at the end so no mask; "How Audio
Becomes Words", "The Full Stitched Circuit": causal self-attention, cross-attention into the
memory, feed-forward, final norm, tied output projection):
- Steps 0..P-1, run one after the other on a growing cache, give the logits of an
  independent full-sequence restatement with torch.nn.functional and a causal
  scaled_dot_product_attention, at every position; the caches hold that restatement's k/v.
- Cache rows past pos are never read (NaN there changes nothing); the step writes row pos
  of every layer's caches and no other row.
- At pos 0 the self-attention has one key: its output is that key's value exactly.
- With every block's output projections zeroed, the logits are the closed form
  E LNf(E[tok] + P[pos]) (the embedding is the output projection).
- The greedy token is the first largest logit.
- Planted mistakes (the token left out of its own attention, positions off by one, the two
  attention norms swapped, the cache row not written) each break the restatement pin.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import whisper_ref as R
from whisper_audio_encoder_gb300 import synth
from whisper_audio_encoder_gb300.configs import EncoderConfig

D, H, L, FF, VOCAB, CAP, NCTX = 128, 2, 2, 512, 300, 16, 37
CFG = EncoderConfig("decode-pin", 80, D, H, L, FF, 1, "sines", index=21)


@pytest.fixture(scope="module")
def setup():
    w = synth.decoder_weights(CFG, n_vocab=VOCAB, n_text_ctx=CAP, ln_random=True)
    kv = synth.cross_kv_values(CFG, 1, NCTX, seed=1)                  # [L][NCTX][2 D]
    xk = [kv[l][:, :D].astype(np.float64) for l in range(L)]
    xv = [kv[l][:, D:].astype(np.float64) for l in range(L)]
    rng = np.random.default_rng(8)
    tokens = rng.integers(0, VOCAB, size=7)
    return w, xk, xv, tokens


def _empty_cache():
    return [np.full((CAP, D), np.nan) for _ in range(L)], [np.full((CAP, D), np.nan) for _ in range(L)]


def _run_steps(w, xk, xv, tokens):
    kc, vc = _empty_cache()
    logits = [R.decode_step(int(t), p, w, kc, vc, xk, xv, H) for p, t in enumerate(tokens)]
    return np.stack(logits), kc, vc


def _torch_decoder(tokens, w, xk, xv):
    """An independent restatement: the whole token sequence at once, causal masking by
    scaled_dot_product_attention(is_causal=True), float64."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    P = len(tokens)
    x = t(w["tok_embd"])[torch.as_tensor(tokens)] + t(w["dec_pos"])[:P]
    heads = lambda a: a.reshape(-1, H, D // H).transpose(0, 1)[None]
    merge = lambda a: a[0].transpose(0, 1).reshape(-1, D)
    ks, vs = [], []
    for l, lw in enumerate(w["layers"]):
        h = F.layer_norm(x, (D,), t(lw["ln1_g"]), t(lw["ln1_b"]), eps=1e-5)
        q, k, v = F.linear(h, t(lw["wq"]), t(lw["bq"])), F.linear(h, t(lw["wk"])), F.linear(h, t(lw["wv"]), t(lw["bv"]))
        ks.append(k.numpy())
        vs.append(v.numpy())
        a = merge(F.scaled_dot_product_attention(heads(q), heads(k), heads(v), is_causal=True))
        x = x + F.linear(a, t(lw["wo"]), t(lw["bo"]))
        h = F.layer_norm(x, (D,), t(lw["lnx_g"]), t(lw["lnx_b"]), eps=1e-5)
        q = F.linear(h, t(lw["xwq"]), t(lw["xbq"]))
        a = merge(F.scaled_dot_product_attention(heads(q), heads(t(xk[l])), heads(t(xv[l]))))
        x = x + F.linear(a, t(lw["xwo"]), t(lw["xbo"]))
        h = F.layer_norm(x, (D,), t(lw["ln2_g"]), t(lw["ln2_b"]), eps=1e-5)
        x = x + F.linear(F.gelu(F.linear(h, t(lw["w1"]), t(lw["b1"]))), t(lw["w2"]), t(lw["b2"]))
    x = F.layer_norm(x, (D,), t(w["lnf_g"]), t(w["lnf_b"]), eps=1e-5)
    return F.linear(x, t(w["tok_embd"])).numpy(), ks, vs


def test_steps_match_the_causal_full_sequence_restatement(setup):
    w, xk, xv, tokens = setup
    got, kc, vc = _run_steps(w, xk, xv, tokens)
    ref, ks, vs = _torch_decoder(tokens, w, xk, xv)
    assert got.shape == (len(tokens), VOCAB)
    assert np.max(np.abs(got - ref)) < 1e-9
    P = len(tokens)
    for l in range(L):
        assert np.max(np.abs(kc[l][:P] - ks[l])) < 1e-12
        assert np.max(np.abs(vc[l][:P] - vs[l])) < 1e-12
        assert np.all(np.isnan(kc[l][P:])) and np.all(np.isnan(vc[l][P:]))   # rows past pos untouched


def test_cache_rows_past_pos_are_never_read(setup):
    w, xk, xv, tokens = setup
    clean, _, _ = _run_steps(w, xk, xv, tokens[:4])
    kc, vc = [np.zeros((CAP, D)) for _ in range(L)], [np.zeros((CAP, D)) for _ in range(L)]
    for p, tok in enumerate(tokens[:4]):
        for l in range(L):                       # garbage past the row this step writes
            kc[l][p:] = np.nan
            vc[l][p:] = np.nan
        out = R.decode_step(int(tok), p, w, kc, vc, xk, xv, H)
        assert np.all(np.isfinite(out))
        np.testing.assert_array_equal(out, clean[p])


def test_first_step_self_attention_is_its_own_value(setup):
    w, _, _, _ = setup
    lw = w["layers"][0]
    rng = np.random.default_rng(9)
    h = rng.standard_normal(D)
    kc, vc = np.zeros((CAP, D)), np.zeros((CAP, D))
    a = R.decoder_self_attention(h, lw, kc, vc, 0, H)
    np.testing.assert_allclose(a, h @ lw["wv"].astype(np.float64).T + lw["bv"], rtol=0, atol=1e-13)
    np.testing.assert_array_equal(a, vc[0])


def test_logits_with_silent_blocks_are_the_tied_closed_form(setup):
    w, xk, xv, _ = setup
    quiet = dict(w)
    quiet["layers"] = [dict(lw, wo=0 * lw["wo"], bo=0 * lw["bo"], xwo=0 * lw["xwo"], xbo=0 * lw["xbo"],
                            w2=0 * lw["w2"], b2=0 * lw["b2"]) for lw in w["layers"]]
    kc, vc = _empty_cache()
    tok, pos = 123, 0
    got = R.decode_step(tok, pos, quiet, kc, vc, xk, xv, H)
    x = w["tok_embd"][tok].astype(np.float64) + w["dec_pos"][pos]
    mu, var = x.mean(), x.var()
    xn = (x - mu) / np.sqrt(var + 1e-5) * w["lnf_g"] + w["lnf_b"]
    np.testing.assert_allclose(got, w["tok_embd"].astype(np.float64) @ xn, rtol=0, atol=1e-12)


def test_greedy_token_is_the_first_maximum():
    assert R.greedy_token(np.array([0.5, 2.0, -1.0, 2.0])) == 1
    assert R.greedy_token(np.array([3.0])) == 0


def test_planted_mistakes_are_caught(setup, monkeypatch):
    """Each plausible slip in the decode step must break the full-sequence restatement."""
    w, xk, xv, tokens = setup
    ref, _, _ = _torch_decoder(tokens[:5], w, xk, xv)

    def worst():
        got, _, _ = _run_steps(w, xk, xv, tokens[:5])
        with np.errstate(invalid="ignore"):
            return np.nanmax(np.abs(got - ref)) if np.all(np.isfinite(got)) else np.inf

    orig_attend, orig_embed, orig_self = R.attend_one, R.decoder_embed, R.decoder_self_attention
    # the token left out of its own self-attention (attends to rows 0..pos-1 only)
    monkeypatch.setattr(R, "attend_one", lambda q, k, v, nh: orig_attend(q, k[:-1], v[:-1], nh)
                        if k.shape[0] < NCTX and k.shape[0] > 1 else orig_attend(q, k, v, nh))
    assert worst() > 1e-3
    monkeypatch.setattr(R, "attend_one", orig_attend)
    # stored positions read one row late
    monkeypatch.setattr(R, "decoder_embed", lambda tok, pos, ww: orig_embed(tok, pos + 1, ww))
    assert worst() > 1e-3
    monkeypatch.setattr(R, "decoder_embed", orig_embed)
    # the self-attention's keys/values attended without this step's row written
    def stale(h, lw, kc, vc, pos, nh):
        k_old, v_old = kc[pos].copy(), vc[pos].copy()
        a = orig_self(h, lw, kc, vc, pos, nh)
        kc[pos], vc[pos] = k_old, v_old
        return a
    monkeypatch.setattr(R, "decoder_self_attention", stale)
    assert worst() > 1e-3
    monkeypatch.setattr(R, "decoder_self_attention", orig_self)
    # the self- and cross-attention norms swapped
    swapped = dict(w, layers=[dict(lw, ln1_g=lw["lnx_g"], ln1_b=lw["lnx_b"], lnx_g=lw["ln1_g"], lnx_b=lw["ln1_b"])
                              for lw in w["layers"]])
    got, _, _ = _run_steps(swapped, xk, xv, tokens[:5])
    assert np.max(np.abs(got - ref)) > 1e-3
