"""GB300-native hot path of Multi-Future Drafting (MFD): LM head + log-softmax
+ top-k, mixture DDTree build, tree verification -- CUDA kernels for sm_103a
behind the C ABI in include/mfd.h, with a thin ctypes binding (``mfd``) and a
seeded synthetic-input generator (``synth``)."""

__all__ = ["mfd", "synth", "build"]
