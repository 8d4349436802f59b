"""B300-native KV-cache importance scoring and rate-distortion compression.

The compute runs in the CUDA library ``libkvs.so`` (C ABI, ``include/kvs.h``);
this package only marshals arguments to it (see ``_lib``) and makes seeded
synthetic inputs (``synth``).
"""
