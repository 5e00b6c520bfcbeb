"""GPU log-mel front end (wh_frontend) against the oracle, element by element, on the
workloads' seeded waveforms (80 and 128 mel bins), plus edge cases: empty, short,
exactly-30-s, long (truncated) and silent clips, and batch-position invariance."""
import numpy as np
import pytest
import torch

from oracle import whisper_ref as R
from whisper_audio_encoder_gb300 import build, configs, synth, wh

from helpers import LOGMEL_ATOL, maxabs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build.build()
    wh.lib()


@pytest.mark.parametrize("idx,windows", [(0, [0]), (1, list(range(8))), (2, [0, 15]), (3, [5, 31]), (4, [0, 15])])
def test_logmel_parity_on_workloads(idx, windows):
    cfg = configs.CONFIGS[idx]
    pcm = synth.waveforms(cfg)                      # the whole batch goes through the kernel
    mel = wh.wh_frontend(torch.from_numpy(pcm).cuda(), cfg.n_mels)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    got = mel.cpu().numpy()
    assert got.shape == (cfg.batch, 3000, cfg.n_mels)
    for w in windows:
        ref = R.log_mel(pcm[w], cfg.n_mels)
        err = maxabs(got[w], ref)
        assert err <= LOGMEL_ATOL, f"window {w}: {err}"
        assert got[w].max() - got[w].min() <= 2.0 + 1e-5


@pytest.mark.parametrize("n", [0, 1, 1000, 144_000, 479_999, 480_000, 480_001, 500_000])
@pytest.mark.parametrize("n_mels", [80, 128])
def test_logmel_lengths(n, n_mels):
    rng = np.random.default_rng(n + n_mels)
    pcm = (0.1 * rng.standard_normal((2, n))).astype(np.float32)
    mel = wh.wh_frontend(torch.from_numpy(pcm).cuda(), n_mels).cpu().numpy()
    for b in range(2):
        ref = R.log_mel(pcm[b], n_mels)
        assert maxabs(mel[b], ref) <= LOGMEL_ATOL, (n, b)
    if n == 0:
        assert np.all(mel == np.float32(-1.5))


def test_silent_and_loud_windows_in_one_batch():
    rng = np.random.default_rng(3)
    pcm = np.zeros((3, 480_000), np.float32)
    pcm[1] = 0.5 * rng.standard_normal(480_000)
    pcm[2, :16000] = 0.01 * rng.standard_normal(16000)
    mel = wh.wh_frontend(torch.from_numpy(pcm).cuda(), 80).cpu().numpy()
    assert np.all(mel[0] == np.float32(-1.5))                  # per-window maximum, not per batch
    for b in (1, 2):
        assert maxabs(mel[b], R.log_mel(pcm[b], 80)) <= LOGMEL_ATOL


def test_batch_position_does_not_change_the_result():
    cfg = configs.CONFIGS[2]
    x = synth.waveform(cfg, 3)
    pcm = np.stack([synth.waveform(cfg, 1), x, synth.waveform(cfg, 2), x])
    mel = wh.wh_frontend(torch.from_numpy(pcm).cuda(), 80).cpu().numpy()
    assert np.array_equal(mel[1], mel[3])


def test_grid_shape_does_not_change_the_result():
    # Alone, the window's 94 tiles each get their own block.  In a batch of 40 windows (3760
    # tiles) every block of the resident grid walks many tiles of several windows and loads
    # each next tile's samples ahead.  Either way each tile is computed the same: bitwise equal.
    cfg = configs.CONFIGS[2]
    x = synth.waveform(cfg, 5)
    alone = wh.wh_frontend(torch.from_numpy(x[None, :].copy()).cuda(), 80).cpu().numpy()[0]
    rng = np.random.default_rng(40)
    pcm = (0.05 * rng.standard_normal((40, 480_000))).astype(np.float32)
    pcm[17] = x
    many = wh.wh_frontend(torch.from_numpy(pcm).cuda(), 80).cpu().numpy()
    assert wh.wh_status() == wh.WH_OK
    assert np.array_equal(alone, many[17])
    assert maxabs(many[39], R.log_mel(pcm[39], 80)) <= LOGMEL_ATOL


@pytest.mark.parametrize("n_mels", [80, 128])
def test_batch_larger_than_the_resident_grid(n_mels):
    # 700 windows: more than the resident grid (about two blocks per SM), so each block's
    # share of the clamp pass covers several whole windows.  Loud and quiet windows alternate
    # (maxima 6 apart in log10), and each is mostly silence, so the clamp at its own
    # maximum - 8 binds; a floor taken from a neighbouring window would show.  Every window
    # must equal, bit for bit, the same window transformed alone.
    rng = np.random.default_rng(700 + n_mels)
    loud = (0.3 * rng.standard_normal(1000)).astype(np.float32)
    quiet = (1e-3 * loud).astype(np.float32)
    batch = 700
    pcm = np.empty((batch, 1000), np.float32)
    pcm[0::2] = loud
    pcm[1::2] = quiet
    pcm[5] = 0.0                                   # one silent window as well
    mel = wh.wh_frontend(torch.from_numpy(pcm).cuda(), n_mels)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    alone = {key: wh.wh_frontend(torch.from_numpy(x[None, :].copy()).cuda(), n_mels)[0]
             for key, x in (("loud", loud), ("quiet", quiet))}
    for key, x in (("loud", loud), ("quiet", quiet)):
        assert maxabs(alone[key].cpu().numpy(), R.log_mel(x, n_mels)) <= LOGMEL_ATOL
    for b in range(batch):
        if b == 5:
            assert bool(torch.all(mel[b] == -1.5)), "silent window"
        else:
            assert torch.equal(mel[b], alone["loud" if b % 2 == 0 else "quiet"]), f"window {b}"
