"""GQA attention over a paged KV cache stored in a 2-bit, 72 B/head/token format.

The compute path lives in ``libkvq.so`` (hand-written CUDA for sm_103a, C ABI declared in
``include/kvq.h``); :mod:`.kvq` is its ctypes binding and :mod:`.synth` the seeded synthetic
workload generator.
"""
