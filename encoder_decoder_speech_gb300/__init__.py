"""GB300-native encoder-decoder cross-attention: projection-cache populate and
split-T decode, behind the C-ABI library ``libcxa`` (see ``include/cxa.h``).

Importing the package loads nothing; ``encoder_decoder_speech_gb300.cxa`` loads
the compiled library on first use and raises if it is missing.
"""
__all__ = ["workloads", "cxa"]
