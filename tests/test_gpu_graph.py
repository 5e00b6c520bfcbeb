"""Recorded passes (wh_graph_capture / wh_graph_launch): a replay gives exactly the memory of
a direct wh_frontend + wh_encode call on the same buffers, also after the PCM is refreshed in
place between replays."""
import numpy as np
import pytest
import torch

from whisper_audio_encoder_gb300 import build, configs, synth, wh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build.build()
    wh.lib()


def test_graph_replay_equals_direct_calls():
    cfg = configs.CONFIGS[1]
    enc = wh.Encoder(cfg, synth.weights(cfg))
    first = torch.from_numpy(synth.waveforms(cfg)).cuda()
    second = torch.from_numpy(synth.waveforms(cfg, windows=range(8, 16))).cuda()
    B = cfg.batch
    pcm = first.clone()
    mel = torch.empty(B, 3000, cfg.n_mels, device="cuda")
    out = torch.empty(B, 1500, cfg.d_model, device="cuda")
    stream = torch.cuda.Stream()
    graph = enc.capture(pcm, mel, out, stream)
    refs = []
    for src in (first, second):
        refs.append(enc.forward(src.clone()).cpu().numpy())
    torch.cuda.synchronize()
    for src, ref in zip((first, second), refs):
        with torch.cuda.stream(stream):
            pcm.copy_(src)
            graph.launch(stream)
        stream.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref)
    assert wh.wh_status() == wh.WH_OK
    graph.destroy()


def test_pipeline_serves_batches_in_order():
    """The double-buffered serving loop (wh.Pipeline) returns, for each of five batches, exactly
    the memory a direct call gives for that batch, although copies and passes overlap."""
    cfg = configs.CONFIGS[1]
    enc = wh.Encoder(cfg, synth.weights(cfg))
    B = cfg.batch
    batches = [torch.from_numpy(synth.waveforms(cfg, windows=range(8 * k, 8 * k + B))).pin_memory()
               for k in range(5)]
    outs = [torch.empty(B, 1500, cfg.d_model).pin_memory() for _ in range(5)]
    pipe = wh.Pipeline(enc, B, batches[0].shape[1])
    pipe.run(batches, outs)
    assert wh.wh_status() == wh.WH_OK
    for k in range(5):
        ref = enc.forward(batches[k].cuda()).cpu()
        torch.cuda.synchronize()
        assert torch.equal(outs[k], ref), f"batch {k}"
    pipe.destroy()


def test_encoder_only_recording_equals_wh_encode():
    cfg = configs.CONFIGS[1]
    enc = wh.Encoder(cfg, synth.weights(cfg))
    mel = wh.wh_frontend(torch.from_numpy(synth.waveforms(cfg)).cuda(), cfg.n_mels)
    ref = enc.wh_encode(mel).clone()
    out = torch.empty_like(ref)
    torch.cuda.synchronize()          # the direct call and the recorded pass share one workspace
    stream = torch.cuda.Stream()
    g = enc.capture_encode(mel, out, stream)
    g.launch(stream)
    stream.synchronize()
    assert torch.equal(out, ref)
    g.destroy()


def test_calls_after_shutdown_set_the_device_up_again():
    cfg = configs.CONFIGS[0]
    x = torch.from_numpy(synth.waveforms(cfg)).cuda()
    a = wh.wh_frontend(x, cfg.n_mels).clone()
    torch.cuda.synchronize()
    assert wh.lib().wh_shutdown() == wh.WH_OK
    b = wh.wh_frontend(x, cfg.n_mels)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    assert torch.equal(a, b)
