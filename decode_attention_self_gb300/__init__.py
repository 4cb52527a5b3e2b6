"""Decode step of a MusicGen-style multi-codebook audio-token decoder on GB300.

The compute lives in a C-ABI CUDA library (``libdecoderattn.so``, sm_103a);
``decode_attention_self_gb300.api`` is its thin ctypes binding.  Importing the
package itself loads nothing, so host-only tools (input generation) work on a
machine without a GPU; importing ``api`` fails loudly when the library is
missing.
"""
__all__ = ["api", "workloads", "build"]
