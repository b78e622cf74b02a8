"""Paged-KV attention over working sets for GB300 (sm_103a).

The library is libpie_attn.so (C ABI in include/pie_attn.h); ``pie`` is its
Python binding, ``build`` compiles it, ``workloads`` makes seeded synthetic
inputs.  Importing this package loads nothing; importing ``pie`` loads the
library.
"""
