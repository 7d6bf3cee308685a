"""CPU oracle for one routed MoE layer forward pass (FP64).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its Python binding) never imports it and shares no code
with it; both only take their inputs from the seeded generator in
``routed_expert_layer_gemv_gb300.workloads``.

What the layer computes.  The FreeToken pages ("FreeToken：把 284B MoE 塞进游戏
PC", zhichai.net, §二; the ananclaw.com explainer, §核心方法 1) describe an
edge MoE serving system whose layers route each token to a few experts held in
a GPU-resident LRU expert cache.  They give no formula for the layer itself,
so the oracle writes out the standard definitions the pages' names refer to:

* ``formats``  E2M1 / E8M0 / E4M3 decoding and MXFP4 / NVFP4 block dequant
  (the formats the pages name: §五 on zhichai.net, §五 of the juejin.cn post);
* ``quant``    the activation quantisers of the FP4 x FP4 prefill regime;
* ``layer``    router (logits, softmax, top-k), permutation, SwiGLU experts,
  gate-weighted combine and the optional shared expert;
* ``lru``      the per-step LRU slot table of the expert cache.

Two implementations of the same definitions:

* ``oracle.native`` -- plain C++ in FP64 (``moe_oracle.cpp``, built by
  ``oracle/build.py`` into ``oracle/_lib/liboracle.so``): fixed-order loops,
  OpenMP over tokens and rows.  This is the oracle the GPU parity tests, the
  smoke check and the bench's CPU baseline use.
* the numpy modules of this package (``formats``, ``quant``, ``layer``,
  ``lru``), kept as a cross-check.

Every function names the passage it follows and, where the pages are silent,
the reading taken.  Parity pins (tests marked ``not gpu``) check each piece of
both implementations against closed forms, library routines and brute force,
and the two against each other.
"""
from . import formats, quant, layer, lru  # noqa: F401
