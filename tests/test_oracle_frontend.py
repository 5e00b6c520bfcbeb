"""Pins of the oracle's front end (log-mel) against things other than itself: closed forms,
invariants, library routines (numpy.fft, torch.stft) and brute force.

Sources: "How Audio Becomes Words: Whisper's Kernels Step By Step On A CPU", section
"The Frontend: Sound Becomes A Tensor" (kernels 3-6: pad/truncate, STFT power with reflect
padding, periodic Hann, n_fft 400, hop 160 to a 201 x 3000 grid; Slaney mel filters,
area-normalised; log10, a global -80 dB clamp and an (x+4)/4 rescale).
"""
import numpy as np
import pytest
import torch

from oracle import whisper_ref as R

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- pad / truncate, framing
def test_pad_or_truncate():
    short = np.arange(10, dtype=np.float32) + 1
    x = R.pad_or_truncate(short)
    assert x.shape == (480_000,) and np.all(x[:10] == short) and np.all(x[10:] == 0)
    long = RNG.standard_normal(500_000)
    assert np.array_equal(R.pad_or_truncate(long), long[:480_000])


def test_frame_grid_is_3000_by_400():
    # 480000 samples, hop 160 -> 3000 frames of 400 samples (the 201 x 3000 grid)
    f = R.frame_signal(np.zeros(480_000))
    assert f.shape == (3000, 400)


def test_reflect_padding_on_a_ramp():
    x = np.arange(480_000, dtype=np.float64)
    f = R.frame_signal(x)
    # frame 0 is centred on sample 0: positions 0..199 mirror samples 200..1 (edge not repeated)
    assert f[0, 200] == 0 and f[0, 199] == 1 and f[0, 0] == 200 and f[0, 201] == 1
    # an interior frame is a plain slice starting at 160 t - 200
    assert np.array_equal(f[1000], x[160_000 - 200: 160_000 + 200])
    # the last frame runs 40 samples past the end: index 480000 reads sample 479998
    last = f[2999]
    start = 160 * 2999 - 200
    assert last[480_000 - start] == 479_998 and last[-1] == 2 * 479_999 - (start + 399)


# ---------------------------------------------------------------- Hann
def test_hann_periodic_closed_form():
    w = R.hann_periodic()
    assert w[0] == 0.0 and w[200] == pytest.approx(1.0, abs=1e-15)
    assert w.sum() == pytest.approx(200.0, abs=1e-9)                 # N/2 for a periodic Hann
    assert np.allclose(w[1:], w[1:][::-1], atol=1e-15)               # w[n] = w[400 - n]
    ref = torch.hann_window(400, periodic=True, dtype=torch.float64).numpy()
    assert np.max(np.abs(w - ref)) < 1e-12


# ---------------------------------------------------------------- DFT power
def test_dft_power_brute_force_vs_numpy_rfft():
    frames = RNG.standard_normal((7, 400))
    w = R.hann_periodic()
    p = R.dft_power(frames, w)
    ref = np.abs(np.fft.rfft(frames * w, axis=1)) ** 2
    assert p.shape == (7, 201)
    assert np.max(np.abs(p - ref)) <= 1e-10 * ref.max()


def test_power_closed_form_single_cosine():
    # x = A cos(2 pi k0 n / 400 * ...) at bin frequency k0 * 40 Hz: an interior frame's
    # periodic-Hann spectrum is exactly three bins: (100 A)^2 at k0, (50 A)^2 at k0 +- 1.
    A = 0.3
    for k0 in (2, 37, 100, 198):
        n = np.arange(480_000)
        x = A * np.cos(2 * np.pi * k0 * 40.0 * n / 16_000 + 0.7)
        p = R.dft_power(R.frame_signal(x)[1500:1503], R.hann_periodic())
        for row in p:
            assert row[k0] == pytest.approx((100 * A) ** 2, rel=1e-9)
            assert row[k0 - 1] == pytest.approx((50 * A) ** 2, rel=1e-9)
            assert row[k0 + 1] == pytest.approx((50 * A) ** 2, rel=1e-9)
            rest = np.delete(row, [k0 - 1, k0, k0 + 1])
            assert rest.max() < 1e-18 * 1e4


def test_stft_power_matches_torch_stft():
    x = RNG.standard_normal(480_000) * 0.1
    p = R.dft_power(R.frame_signal(R.pad_or_truncate(x)), R.hann_periodic())
    st = torch.stft(torch.from_numpy(x), n_fft=400, hop_length=160,
                    window=torch.hann_window(400, periodic=True, dtype=torch.float64),
                    center=True, pad_mode="reflect", return_complex=True)
    ref = (st.abs() ** 2).numpy().T[:3000]          # torch gives 3001 frames; the grid has 3000
    assert ref.shape == p.shape == (3000, 201)
    assert np.max(np.abs(p - ref)) <= 1e-10 * ref.max()


# ---------------------------------------------------------------- Slaney mel filterbank
def test_slaney_scale_closed_forms():
    assert R.hz_to_mel_slaney(0.0) == 0.0
    assert R.hz_to_mel_slaney(200.0) == pytest.approx(3.0)
    assert R.hz_to_mel_slaney(1000.0) == pytest.approx(15.0)
    assert R.hz_to_mel_slaney(6400.0) == pytest.approx(42.0)          # 15 + 27 per factor 6.4
    assert R.hz_to_mel_slaney(6400.0 * 6.4) == pytest.approx(69.0)
    f = np.array([0.0, 40.0, 999.0, 1000.0, 1001.0, 4321.0, 8000.0])
    assert np.allclose(R.mel_to_hz_slaney(R.hz_to_mel_slaney(f)), f, rtol=1e-12, atol=1e-9)
    # continuous at the 1 kHz knee
    assert R.hz_to_mel_slaney(1000.0 - 1e-9) == pytest.approx(R.hz_to_mel_slaney(1000.0), abs=1e-9)


@pytest.mark.parametrize("n_mels", [80, 128])
def test_mel_filterbank_structure(n_mels):
    fb = R.mel_filterbank(n_mels)
    assert fb.shape == (n_mels, 201)
    assert np.all(fb >= 0)
    assert np.all((fb > 0).sum(axis=0) <= 2)                          # each bin in <= 2 triangles
    assert np.all((fb > 0).sum(axis=1) >= 1)                          # no empty filter
    assert np.all(np.diff(np.argmax(fb, axis=1)) >= 0)                # ordered by centre
    edges = R.mel_to_hz_slaney(np.linspace(0, R.hz_to_mel_slaney(8000.0), n_mels + 2))
    assert np.all(fb.max(axis=1) <= 2.0 / (edges[2:] - edges[:-2]) + 1e-15)


@pytest.mark.parametrize("n_mels", [80, 128])
def test_mel_filterbank_is_area_normalised_triangles(n_mels):
    fb = R.mel_filterbank(n_mels)
    edges = R.mel_to_hz_slaney(np.linspace(0, R.hz_to_mel_slaney(8000.0), n_mels + 2))
    bins = np.arange(201) * 40.0
    for m in range(n_mels):
        lo, c, hi = edges[m], edges[m + 1], edges[m + 2]
        tri = np.interp(bins, [lo, c, hi], [0.0, 2.0 / (hi - lo), 0.0], left=0.0, right=0.0)
        assert np.max(np.abs(fb[m] - tri)) < 1e-12
    # un-normalised triangles form a partition of unity between the first and last centre
    unnorm = (fb * ((edges[2:] - edges[:-2]) / 2.0)[:, None]).sum(axis=0)
    inside = (bins >= edges[1]) & (bins <= edges[-2])
    assert np.allclose(unnorm[inside], 1.0, atol=1e-12)
    # area of a wide triangle (height 2/base, base >= 10 bins) is ~1 (Riemann sum at 40 Hz)
    wide = (edges[2:] - edges[:-2]) >= 400.0
    area = fb.sum(axis=1) * 40.0
    assert np.allclose(area[wide], 1.0, atol=0.02)


# ---------------------------------------------------------------- log-mel
def test_log_mel_all_zero_window_is_minus_1_5():
    mel = R.log_mel(np.zeros(480_000, np.float32), 80)
    assert mel.shape == (3000, 80) and np.all(mel == np.float32(-1.5))


def test_log_mel_empty_input_is_silence():
    assert np.all(R.log_mel(np.zeros(0, np.float32), 128) == np.float32(-1.5))


@pytest.mark.parametrize("silent_tail", [False, True])
def test_log_mel_clamp_invariants(silent_tail):
    x = (RNG.standard_normal(480_000) * 0.05).astype(np.float32)
    if silent_tail:
        x[144_000:] = 0.0
    fb = R.mel_filterbank(80)
    p = R.dft_power(R.frame_signal(R.pad_or_truncate(x)), R.hann_periodic())
    s = p @ fb.T
    mel = R.log_mel(x, 80).astype(np.float64)
    g = np.log10(s.max())
    assert mel.max() == pytest.approx((g + 4) / 4, abs=1e-6)
    assert mel.max() - mel.min() <= 2.0 + 1e-6
    if silent_tail:      # silent frames sit exactly on the floor: the clamp binds
        assert mel.max() - mel.min() == pytest.approx(2.0, abs=1e-6)
        assert np.all(mel[1000:] == mel.min())


def test_log_mel_matches_torch_restatement():
    x = (RNG.standard_normal(300_000) * 0.1).astype(np.float32)       # short clip: zero-padded
    xt = torch.zeros(480_000, dtype=torch.float64)
    xt[:300_000] = torch.from_numpy(x.astype(np.float64))
    st = torch.stft(xt, 400, 160, window=torch.hann_window(400, periodic=True, dtype=torch.float64),
                    center=True, pad_mode="reflect", return_complex=True)[:, :3000]
    s = torch.from_numpy(R.mel_filterbank(80)) @ (st.abs() ** 2)
    lg = torch.log10(torch.clamp(s, min=1e-10))
    lg = torch.maximum(lg, lg.max() - 8.0)
    ref = ((lg + 4.0) / 4.0).T.numpy()
    assert np.max(np.abs(R.log_mel(x, 80) - ref)) < 1e-6
