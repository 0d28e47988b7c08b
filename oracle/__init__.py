"""CPU oracle for the W4A16 NVFP4 weight-only GEMM -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the
weight-only NVFP4 path computes, written in numpy (float64 wherever the
sources leave the precision open).  It exists to check the CUDA library, never
to stand in for it: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import it.  The product path
(``w4a16_nvfp4_weight_gb300``) never imports it and shares no code, table or
helper with it.

Sources (cited by page title and section):

* "[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt on Hopper"
  (TensorRT-LLM PR 14775), Walkthrough/Changes table: the dequant is an
  "E2M1 FP4 codebook lookup" with "per-block FP8 scale conversion" and a
  per-tensor scale (2D path); the MoE path dequantizes only active experts and
  then runs a BF16 fused MoE; the linear path runs a BF16 GEMM on the
  dequantized weight.
* SGLang PR 40022 (compressed-tensors NVFP4 served weight-only), Motivation and
  Modifications: group size 16, E4M3 group scales, a real per-tensor global
  scale, and the global stored as a divisor that must be inverted first.
* "[None][fix] Apply the NVFP4_AWQ pre-quant scale in MegaMoE CuteDSL"
  (TensorRT-LLM PR 20823), Description and commit messages: stored weights are
  W/s so the activation must be x*s, shape [1, hidden], the product kept in
  BF16; a zero-token chunk launches nothing.

Modules:

* ``formats``  -- E2M1 / E4M3 decoding, global-scale inversion, BF16 rounding.
* ``dense``    -- dequantization, AWQ activation scaling, the GEMM.
* ``moe``      -- top-k routing, permutation tables, FC1+SwiGLU, FC2, combine.

Parity status of every function is stated in its docstring; every function is
pinned by ``tests/test_oracle_*.py`` against worked values, closed forms,
library routines or brute force on tiny inputs.
"""

from . import formats, dense, moe  # noqa: F401
