"""CPU oracle for the fused 4-bit block-scaled MoE layer.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and
its Python binding) imports, links or runs this package; only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` do.

It is a plain, slow, obviously-correct restatement of what the layer computes,
written in NumPy with float64 accumulation. Formats are decoded through
explicit tables built from their definitions; no code is shared with the CUDA
sources under ``bit_block_scaled_gb300/csrc``.

Sources (web pages on the subject, cited by title and section):
  * vLLM issue "moe_wna16_marlin_gemm applies wrong per-row topk weights
    (mul_topk_weights=True) at gpt-oss NVFP4 MoE shapes" -- "Minimal repro":
    E2M1 value table, packed-nibble order, NVFP4 dequant formula, fp32
    per-row reference ``(act[row] @ w[e].T + bias) * topk_w[row]``, the
    alignment metadata and the per-row applied-ratio forensic.
  * vLLM issue "gpt-oss-20b NVFP4 inference is broken" -- Gaps 1, 2, 3c:
    per-expert biases, per-expert global scale, interleaved gate/up rows,
    clamped SwiGLU ("swigluoai").
  * vLLM issue "NVFP4 MoE monolithic backend ... non-gated ReLU2 MoE
    (Nemotron-3-Nano)" -- Environment and Analysis item 3: non-gated ReLU2
    experts, sigmoid+bias grouped top-k with n_group=1, group size 16.
  * vLLM issue "gpt-oss-120b MXFP4 + --enable-expert-parallel crashes" --
    Root cause: the layer output is [T, H] at the unpadded hidden size.
  * OneCompression guide "GPT-OSS (mixed_gptq)" -- "Why GPT-OSS needs special
    handling" and "1. Quantize": GPTQ INT4 experts with group_size 64.

Parity status per function is listed in each module's header.
"""
from . import formats, routing, align, layer  # noqa: F401
