"""wh_frontend_static -- the front end for callers that cannot allocate device memory (a
real-time audio callback that must not block on the CUDA allocator, or a process whose
device memory is all owned by another allocator) -- must give the same log-mel as
wh_frontend, which takes a caller-allocated scratch buffer.

Called through the C ABI twice in a row, with different batches, so that state left in the
library's fixed scratch array by the first call would show in the second.  This file is
collected last and also passes when run alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import whisper_ref as R
from whisper_audio_encoder_gb300 import build, wh

from helpers import LOGMEL_ATOL, maxabs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build.build()
    return wh.lib()


def _static(L, pcm, n_mels):
    batch, n = pcm.shape
    mel = torch.empty(batch, 3000, n_mels, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.wh_frontend_static(ctypes.c_void_p(pcm.data_ptr()), n, batch, n_mels, ctypes.c_void_p(mel.data_ptr()),
                              stream)
    assert rc == wh.WH_OK, wh.wh_strerror(rc)
    return mel


def test_static_scratch_front_end_matches_workspace_front_end(L):
    # Both entry points run the same kernel, so they must agree bit for bit; a slip in how
    # the fixed scratch array is cleared or addressed between calls would show as a
    # difference.  One window of each call is also checked against the oracle.
    rng = np.random.default_rng(2024)
    loud = (0.3 * rng.standard_normal((5, 480_000))).astype(np.float32)
    quiet = (1e-3 * rng.standard_normal((3, 200_000))).astype(np.float32)   # a much lower maximum
    quiet[1] = 0.0                                                          # and a silent window
    for pcm_np, n_mels in ((loud, 128), (quiet, 80)):                       # two calls in a row
        pcm = torch.from_numpy(pcm_np).cuda()
        ref = wh.wh_frontend(pcm, n_mels)                                  # caller-allocated scratch
        got = _static(L, pcm, n_mels)
        torch.cuda.synchronize()
        assert wh.wh_status() == wh.WH_OK
        assert torch.equal(got, ref)
        assert maxabs(got[0].cpu().numpy(), R.log_mel(pcm_np[0], n_mels)) <= LOGMEL_ATOL
    assert bool(torch.all(got[1] == -1.5))


def test_static_front_end_rejects_batches_beyond_its_scratch(L):
    limit = 4096                                     # WH_FRONTEND_STATIC_MAX_BATCH
    fake = ctypes.c_void_p(1 << 20)                  # rejected before any use
    assert L.wh_frontend_static(fake, 480_000, limit + 1, 80, fake, None) == wh.WH_ENOSPC
    assert L.wh_frontend_static(fake, 480_000, 1, 81, fake, None) == wh.WH_EINVAL
