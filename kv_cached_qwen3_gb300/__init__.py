"""GB300-native KV-cached Qwen3 Talker decoder forward.

The compute runs in the CUDA library built from ``csrc/`` (C-ABI declared in
``include/talker.h``); ``talker`` is its thin ctypes binding and ``inputs`` the
seeded synthetic input generator. Nothing is imported eagerly, so importing the
package never loads the CUDA library.
"""
__all__ = ["inputs", "talker"]
