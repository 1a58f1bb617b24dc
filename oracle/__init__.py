"""CPU oracle for the fused NVFP4 Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, deliberately
unoptimised restatement of what the layer computes. It exists to check the
CUDA path; it is not part of it. Only the tests, the smoke check of the build
entry point and the benchmark's CPU-baseline leg may import it. The CUDA
library and its Python binding never import it, and it imports nothing from
them: the two share no code, tables or helpers.

Sources (web pages, cited by title and section):

* "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 6.1
  (NVFP4 format: e2m1 elements packed two per byte, one FP8-E4M3 scale per 16
  elements along K, one fp32 global scale per tensor, alpha =
  1/(input_global_scale * weight_global_scale)); section 4.3 (the fused MoE
  kernel: token dispatch, two GEMMs, SwiGLU, top-k weight reduction, BF16
  input quantised to FP4 inside the kernel); section 7.1 (router ->
  quantise-dispatch -> permute-experts-unpermute -> combine).
* "Serving Solar Open 2 on DGX Spark", sections "Solar Open 2 in brief"
  (routed experts plus one shared expert, top-k routing) and "Supporting real
  NVFP4 checkpoints" (FP8 block scales re-rounded with a clamp at 448).
* "GLM-5.3-Flash-NVFP4 #4" discussion, the follow-up on the MoE fault (the
  global scale is a reciprocal: dequant scale amax/(448*6) versus quant scale
  (448*6)/amax; worked value 4.650297705666162e-05 against 21504.0).
* the same guide, section 6.4 (MXFP4: e2m1 elements, blocks of 32, E8M0
  scales), for ``mxfp4``.

Precision: everything is float64 except the quantiser, whose decisions are
integer codes and are therefore taken in fp32 with correctly rounded IEEE
operations, the precision the CUDA kernels use.

Parity status of each function is stated in its docstring ("pinned by ...").
"""
from . import nvfp4, moe, mxfp4  # noqa: F401
