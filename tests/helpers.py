"""Comparison helpers and tolerances shared by the GPU parity tests.

Tolerances (stated for bf16 tensor-core operands with fp32 accumulation):
  log-mel            max |gpu - oracle| <= 1e-3
  encoder output     max |gpu - oracle| <= 3e-2 and cosine(gpu frame, oracle frame) >= 0.999
                     for every frame of every compared window
  stand-alone attention with a peaked softmax (q, k ~ N(0, 1)): max |O - O_ref| <= 1e-2
"""
import numpy as np

LOGMEL_ATOL = 1e-3
ENC_ATOL = 3e-2
ENC_MIN_COS = 0.999
ATTN_ATOL = 1e-2


def maxabs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


def frame_cosines(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    num = (a * b).sum(axis=-1)
    den = np.linalg.norm(a, axis=-1) * np.linalg.norm(b, axis=-1)
    return num / np.maximum(den, 1e-300)


def check_encoder(out, ref, what=""):
    err = maxabs(out, ref)
    cmin = float(frame_cosines(out, ref).min())
    assert err <= ENC_ATOL and cmin >= ENC_MIN_COS, f"{what}: max-abs {err:.3e}, min frame cosine {cmin:.6f}"
    return err, cmin


def bf16_round_np(a):
    """Round to bfloat16 (nearest even) and widen back, numpy only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    u = (u + (((u >> 16) & 1) + np.uint32(0x7FFF))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)
