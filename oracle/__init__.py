"""CPU oracle for the hybrid W4A16 mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``nf3_moe_gb300``) never imports it, and it imports
nothing from the product: the two share no code, headers or tables.

It is plain and slow on purpose. NumPy float64 is used throughout. Each
function names the passage of the pages it follows.

The pages are three pull requests:
  [P1] "quant: nvfp4_nf3_hybrid — native serving for mixed NVFP4+NF3 MoE
       checkpoints" (local-inference-lab/vllm #92)
  [P2] "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE serving" (#104)
  [P3] "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE +
       --override-activation-dtype flag" (vllm-project/vllm #42428)

The pages leave every numeric definition open: codebook, group sizes, scale
layouts, routing function. The readings taken here are those written out in
the repository's design notes. Each module header states its own.

Modules:
  formats -- element and scale decoders (E2M1, E4M3, E8M0, NF3 codebook,
             bf16 and fp16 rounding) and dequantisation of the logical checkpoint
             layouts.
  route   -- top-k routing, renormalised gates, stable permutation, offsets.
  layer   -- the SwiGLU expert layer: dequantise, then matmul, gate, sum.
  linear  -- the dense-Linear W4A16 product: dequantise, then matmul.
  actquant -- NVFP4 activation quantisation (the W4A4 layer's x and h).

Every function here is pinned by ``tests/test_oracle_*.py`` against library
routines, closed forms, golden fixtures or brute force.
"""

from . import formats, route, layer, linear, actquant  # noqa: F401
