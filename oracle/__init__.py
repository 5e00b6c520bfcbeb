"""CPU oracle of the Whisper audio-encoder path: test infrastructure only (see whisper_ref)."""
