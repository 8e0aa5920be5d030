"""GB300-native per-frame streaming decode step of the Moshi/PersonaPlex temporal
transformer and depformer.

The compute path is the C-ABI library `libpm` (hand-written sm_103a CUDA);
`full_duplex_speech_moshi_gb300.pm` is its thin ctypes binding.  `inputs` holds the
seeded synthetic inputs.  Nothing here is imported eagerly.
"""
__all__ = ["pm", "inputs"]
