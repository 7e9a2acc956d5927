"""CPU reference ("oracle") for the paged MoE layer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only the test-suite, the smoke check in ``__graft_entry__`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library and imports nothing from it.

Sources (the pages this follows):

* "Paged Experts" (SGLang docs): the K-slot table and host store, the step
  (waves of at most K distinct experts, resident first; LRU eviction outside
  the wave; page-in; remap to slots; the MoE kernel without its top-k sum,
  output already times the router weight; one merged buffer; the same top-k
  sum), captured decode, and the correctness claim (paged output equals
  unpaged output).
* "SGLang Paged Experts: corré MoE más grandes que tu VRAM" (blog.donweb.com):
  model geometry (48 MoE layers, top-8 of 128 experts), per-expert byte sizes
  and the miss-rate arithmetic used as worked examples in the tests, and the
  MXFP4 / NVFP4 formats with their padding lesson.

Everything floating-point here is computed in float64, from the storage
formats (bf16 bits, E4M3 codes with fp32 scales, GPTQ int4 codes with fp16
group scales, E2M1 codes with E8M0 or E4M3 block scales, fp32 router
logits).  Where
the pages are silent the plainest reading is taken; each such reading is
listed in the function that makes it.

Modules:
  routing  softmax over E, top-k on the logits, renormalised weights
  fp8      E4M3 decoding and 128x128 block dequantisation
  int4     GPTQ int4 codes, group-128 dequantisation, checkpoint layout
  fp4      E2M1 codes, MXFP4 (E8M0 per 32) and NVFP4 (E4M3 per 16, fp32
           per tensor) dequantisation
  mlp      SiLU-gated expert MLP, merged buffer, top-k sum, whole layer
  lru      the LRU residency simulator that defines plans, slots and counts
"""

from . import fp4, fp8, int4, lru, mlp, routing  # noqa: F401
