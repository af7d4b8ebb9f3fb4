"""GB300-native MosaicKV decode-time hot path (packed two-D compressed KV cache).

The compute lives in ``libmosaickv.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/mosaickv.h``).  ``binding`` wraps it with ctypes;
``synth`` makes seeded inputs; ``configs`` lists the workloads.
"""
