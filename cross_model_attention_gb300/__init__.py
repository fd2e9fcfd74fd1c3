"""GB300-native hot path of cross-model attention-map reuse (MapFlow-style).

The compute path lives in ``libmapflow.so`` (CUDA, sm_103a) behind a C ABI;
:mod:`cross_model_attention_gb300.mapflow` is the thin ctypes binding.
"""
