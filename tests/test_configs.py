"""The five workloads follow the Whisper family table printed on the pages
(tests/golden/whisper_family.txt), and their flop counts follow from the shapes."""
import os

import pytest

from whisper_audio_encoder_gb300.configs import CONFIGS, N_CTX, N_FRAMES, N_SAMPLES

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "whisper_family.txt")


def _family():
    rows = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if line:
            rows[line[0]] = tuple(int(v) for v in line[1:])
    return rows


@pytest.mark.parametrize("cfg,name", [(CONFIGS[1], "tiny"), (CONFIGS[2], "base"),
                                      (CONFIGS[3], "small"), (CONFIGS[4], "large-v3")])
def test_configs_follow_the_family_table(cfg, name):
    layers, d, heads, mels = _family()[name]
    assert (cfg.n_layer, cfg.d_model, cfg.n_head, cfg.n_mels) == (layers, d, heads, mels)
    assert cfg.d_ff == 4 * cfg.d_model and cfg.head_dim == 64


def test_fixed_geometry():
    assert N_SAMPLES == 30 * 16000 and N_FRAMES == N_SAMPLES // 160 and N_CTX == N_FRAMES // 2
    c0 = CONFIGS[0]
    assert (c0.n_layer, c0.d_model, c0.n_head, c0.batch) == (1, 384, 6, 1)


def test_flops_per_window_large_v3():
    f = CONFIGS[4].flops_per_window()
    assert f["total"] == pytest.approx(2273.8e9, rel=1e-3)
    assert f["attn"] / f["total"] == pytest.approx(0.162, abs=0.002)
