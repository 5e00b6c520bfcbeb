"""GPU parity of the decoder step (wh_decode_step, called through the C ABI) against the
oracle's decode_step, on the same seeded weights, cross-attention keys/values and tokens.

Tolerances (bf16 tensor-core operands, fp32 accumulation and residual stream):
- logits of every sequence: the encoder bar, max |gpu - oracle| <= 3e-2 and cosine >= 0.999
  (the logit vector plays the role of an output frame);
- the greedy token equals the argmax of the GPU's own logits (the same fp32 values decide
  it, first index on a tie), and the oracle's argmax wherever its top two logits are further
  apart than twice the logit tolerance;
- the self-attention cache rows the step writes: |gpu - oracle| <= 2^-7 |oracle| + 1e-2
  (bf16 storage, 2^-9, plus the bf16 rounding of the LayerNorm output feeding the
  projection, summed over d terms).
Cases: several consecutive steps on a growing cache (tiny width, a vocabulary that is not a
multiple of 128, 37 encoder positions); ragged positions with NaN in every cache row past a
sequence's position (never read); large-v3 width (d 1280, 20 heads, vocabulary 51866, 1500
encoder positions, 16 sequences); the full 32-layer large-v3 decoder on sampled sequences;
batches of 1, 17 and 256 sequences; out-of-range tokens and positions (WH_EBOUNDS, clamped);
bitwise repeatability; a recorded step replayed.
"""
import numpy as np
import pytest
import torch

from oracle import whisper_ref as R
from whisper_audio_encoder_gb300 import build, configs, synth, wh
from whisper_audio_encoder_gb300.configs import EncoderConfig

from helpers import ENC_ATOL, ENC_MIN_COS, frame_cosines, maxabs

pytestmark = pytest.mark.gpu

LOGIT_ATOL, LOGIT_MIN_COS = ENC_ATOL, ENC_MIN_COS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build.build()
    wh.lib()


def _bf16_nan():
    return torch.tensor(float("nan"), dtype=torch.bfloat16)


class Case:
    """One decoder, B sequences, their cross K/V and caches on both sides."""

    def __init__(self, cfg, n_layer, n_vocab, cap, batch, n_ctx, seed=0):
        self.cfg, self.B, self.n_ctx, self.cap, self.H = cfg, batch, n_ctx, cap, cfg.n_head
        self.w = synth.decoder_weights(cfg, n_layer=n_layer, n_vocab=n_vocab, n_text_ctx=cap, ln_random=True)
        self.L, self.d = n_layer, cfg.d_model
        kv = synth.cross_kv_values(cfg, batch, n_ctx, n_layer=n_layer, seed=seed)   # [L][B n_ctx][2 d]
        self.kv_dev = torch.from_numpy(kv).to(torch.bfloat16).cuda()
        kv = kv.reshape(n_layer, batch, n_ctx, 2 * self.d).astype(np.float64)
        self.xk = [[kv[l, b, :, :self.d] for l in range(n_layer)] for b in range(batch)]
        self.xv = [[kv[l, b, :, self.d:] for l in range(n_layer)] for b in range(batch)]
        self.dec = wh.Decoder(self.H, self.w, batch)
        self.dec.kcache.fill_(_bf16_nan())                 # nothing past a sequence's position is read
        self.dec.vcache.fill_(_bf16_nan())
        self.kc = [[np.full((cap, self.d), np.nan) for _ in range(n_layer)] for _ in range(batch)]
        self.vc = [[np.full((cap, self.d), np.nan) for _ in range(n_layer)] for _ in range(batch)]

    def prefill(self, rows, seed=1):
        """Rows 0 .. rows[b]-1 of every layer's caches get the same bf16 values on both sides."""
        rng = np.random.default_rng(seed)
        for b, n in enumerate(rows):
            for l in range(self.L):
                for cache, host in ((self.dec.kcache, self.kc), (self.dec.vcache, self.vc)):
                    vals = synth.bf16_round((0.7 * rng.standard_normal((n, self.d))).astype(np.float32))
                    cache[l, b, :n] = torch.from_numpy(vals).to(torch.bfloat16)
                    host[b][l][:n] = vals

    def step(self, tokens, positions):
        tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
        pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
        logits, nxt = self.dec.wh_decode_step(tok, pos, self.kv_dev, self.n_ctx)
        torch.cuda.synchronize()
        st = wh.wh_status()
        return logits.cpu().numpy(), nxt.cpu().numpy(), st

    def oracle(self, b, token, position):
        return R.decode_step(int(token), int(position), self.w, self.kc[b], self.vc[b], self.xk[b], self.xv[b],
                             self.H)

    def check(self, b, got, ref, nxt, what):
        err = maxabs(got, ref)
        cos = float(frame_cosines(got[None], ref[None])[0])
        assert err <= LOGIT_ATOL and cos >= LOGIT_MIN_COS, f"{what}: max-abs {err:.3e}, cosine {cos:.6f}"
        assert np.all(np.isfinite(got)), what
        assert nxt == int(np.argmax(got)), what                      # same fp32 values decide it
        top = np.sort(ref)[-2:]
        if top[1] - top[0] > 2 * LOGIT_ATOL:
            assert nxt == R.greedy_token(ref), what

    def check_cache_rows(self, b, position, what):
        for l in range(self.L):
            for cache, host in ((self.dec.kcache, self.kc), (self.dec.vcache, self.vc)):
                got = cache[l, b, position].float().cpu().numpy()
                ref = host[b][l][position]
                bad = np.abs(got - ref) > 2.0 ** -7 * np.abs(ref) + 1e-2
                assert not bad.any(), f"{what}: layer {l} cache row {position}: {bad.sum()} outside"


TINY = EncoderConfig("dec-tiny", 80, 384, 6, 2, 1536, 3, "sines", index=31)


def test_consecutive_steps_on_a_growing_cache():
    c = Case(TINY, n_layer=2, n_vocab=2000, cap=24, batch=3, n_ctx=37)
    rng = np.random.default_rng(5)
    toks = rng.integers(0, 2000, size=(5, 3))
    for p in range(5):
        got, nxt, st = c.step(toks[p], [p] * 3)
        assert st == wh.WH_OK
        for b in range(3):
            ref = c.oracle(b, toks[p][b], p)
            c.check(b, got[b], ref, nxt[b], f"step {p}, sequence {b}")
            c.check_cache_rows(b, p, f"step {p}, sequence {b}")


def test_ragged_positions_never_read_past_their_row():
    c = Case(TINY, n_layer=2, n_vocab=2000, cap=24, batch=4, n_ctx=37, seed=3)
    positions = [0, 3, 11, 23]                     # 23: the last row of the caches
    c.prefill(positions)
    toks = [7, 1999, 0, 1234]
    got, nxt, st = c.step(toks, positions)
    assert st == wh.WH_OK
    for b in range(4):
        c.check(b, got[b], c.oracle(b, toks[b], positions[b]), nxt[b], f"sequence {b} at {positions[b]}")
        c.check_cache_rows(b, positions[b], f"sequence {b}")


def test_large_v3_width():
    cfg = configs.CONFIGS[4]
    c = Case(cfg, n_layer=2, n_vocab=cfg.n_vocab, cap=448, batch=16, n_ctx=1500, seed=4)
    positions = [int(p) for p in np.linspace(0, 300, 16)]
    c.prefill(positions, seed=2)
    rng = np.random.default_rng(6)
    for k in range(2):
        toks = rng.integers(0, cfg.n_vocab, size=16)
        pos = [p + k for p in positions]
        got, nxt, st = c.step(toks, pos)
        assert st == wh.WH_OK
        for b in (0, 5, 15) if k == 0 else range(16):
            c.check(b, got[b], c.oracle(b, toks[b], pos[b]), nxt[b], f"step {k}, sequence {b}")
        if k == 0:                                  # keep the oracle caches of the others in step
            for b in set(range(16)) - {0, 5, 15}:
                c.oracle(b, toks[b], pos[b])


def test_full_large_v3_decoder_sampled_sequences():
    cfg = configs.CONFIGS[4]
    c = Case(cfg, n_layer=cfg.n_layer, n_vocab=cfg.n_vocab, cap=448, batch=16, n_ctx=1500, seed=7)
    toks = np.random.default_rng(8).integers(0, cfg.n_vocab, size=16)
    got, nxt, st = c.step(toks, [0] * 16)
    assert st == wh.WH_OK
    for b in (0, 15):
        c.check(b, got[b], c.oracle(b, toks[b], 0), nxt[b], f"32 layers, sequence {b}")


def test_out_of_range_tokens_and_positions_are_clamped_and_reported():
    c = Case(TINY, n_layer=1, n_vocab=500, cap=16, batch=4, n_ctx=20, seed=9)
    c.prefill([15, 15, 15, 15])
    kc0, vc0 = c.dec.kcache.clone(), c.dec.vcache.clone()
    assert wh.wh_status() == wh.WH_OK
    got, nxt, st = c.step([-1, 500, 3, 4], [16, -5, 2, 15])
    assert st == wh.WH_EBOUNDS
    assert wh.wh_status() == wh.WH_OK                  # read and cleared
    c.dec.kcache.copy_(kc0)
    c.dec.vcache.copy_(vc0)
    ref, nref, st = c.step([0, 499, 3, 4], [15, 0, 2, 15])
    assert st == wh.WH_OK
    assert np.array_equal(got, ref) and np.array_equal(nxt, nref)


def test_repeated_step_is_bitwise_identical():
    c = Case(TINY, n_layer=2, n_vocab=2000, cap=24, batch=3, n_ctx=37, seed=10)
    c.prefill([4, 9, 2])
    a, na, _ = c.step([1, 2, 3], [4, 9, 2])
    b, nb, _ = c.step([1, 2, 3], [4, 9, 2])           # rewrites the same cache rows
    assert np.array_equal(a, b) and np.array_equal(na, nb)


def test_recorded_step_replays_the_direct_call_and_follows_new_tokens():
    """wh_graph_capture_decode: a replay gives the direct call's logits bit for bit, and
    reads tok / pos afresh at every replay (a decode loop refreshes them in place)."""
    c = Case(TINY, n_layer=2, n_vocab=2000, cap=24, batch=3, n_ctx=37, seed=11)
    c.prefill([3, 3, 3])
    tok = torch.tensor([5, 6, 7], dtype=torch.int32, device="cuda")
    pos = torch.tensor([3, 3, 3], dtype=torch.int32, device="cuda")
    k0, v0 = c.dec.kcache.clone(), c.dec.vcache.clone()
    ref = [c.dec.wh_decode_step(tok, pos, c.kv_dev, c.n_ctx)[0].clone()]
    tok2 = c.dec.next_tok.clone()
    pos.add_(1)
    ref.append(c.dec.wh_decode_step(tok2, pos, c.kv_dev, c.n_ctx)[0].clone())
    c.dec.kcache.copy_(k0)
    c.dec.vcache.copy_(v0)
    pos.fill_(3)
    s = torch.cuda.Stream()
    graph = c.dec.capture(tok, pos, c.kv_dev, c.n_ctx, s)
    graph.launch(s)
    s.synchronize()
    assert torch.equal(c.dec.logits, ref[0])
    with torch.cuda.stream(s):
        tok.copy_(c.dec.next_tok)
        pos.add_(1)
    graph.launch(s)
    s.synchronize()
    assert torch.equal(c.dec.logits, ref[1])
    graph.destroy()
    assert wh.wh_status() == wh.WH_OK


@pytest.mark.parametrize("batch", [1, 17, 256])
def test_batch_sizes_from_one_to_the_maximum(batch):
    """One sequence; 17 (one past a 16-row MMA column block, so the padded rows of the
    operand are live); 256, the largest batch (a full 256-column accumulator)."""
    c = Case(TINY, n_layer=1, n_vocab=700, cap=12, batch=batch, n_ctx=9, seed=12 + batch)
    rng = np.random.default_rng(batch)
    positions = rng.integers(0, 12, size=batch)
    c.prefill(positions, seed=batch)
    toks = rng.integers(0, 700, size=batch)
    got, nxt, st = c.step(toks, positions)
    assert st == wh.WH_OK
    for b in sorted({0, batch // 2, batch - 1}):
        c.check(b, got[b], c.oracle(b, toks[b], positions[b]), nxt[b], f"batch {batch}, sequence {b}")
        c.check_cache_rows(b, positions[b], f"batch {batch}, sequence {b}")
