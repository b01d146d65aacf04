"""GB300-native OSCAR-style rotated INT2 KV cache: append + split-K decode attention.

The compute lives in ``liboscar.so`` (CUDA for sm_103a + a C ABI, see
``include/oscar.h``); ``rotated_int2_kv_gb300.ops`` is a thin ctypes binding
over it, and ``rotated_int2_kv_gb300.synth`` draws seeded synthetic inputs.
"""
