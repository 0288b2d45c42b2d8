"""libfattn: exact tiled attention (FlashAttention forward with online
softmax, recompute backward) as hand-written sm_103a kernels behind a C ABI.

``exact_attention_93_gb300.fattn`` is the ctypes binding to ``libfattn.so``;
``exact_attention_93_gb300.workloads`` draws seeded synthetic inputs.  Import
the submodule you need; importing the package itself loads neither, so that
drawing inputs needs no built library.
"""
