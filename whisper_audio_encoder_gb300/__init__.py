"""GB300-native Whisper audio encoder: log-mel front end + conv stem + pre-LN transformer
encoder as hand-written sm_103a CUDA kernels behind a small C ABI (libwh.so).

`whisper_audio_encoder_gb300.wh` is the Python binding of that ABI (ctypes; torch tensors
are used for device memory and streams only).  Importing this package does not load the
CUDA library; the binding loads it on first use and raises if it has not been built.
"""
__all__ = ["configs", "synth", "wh"]
