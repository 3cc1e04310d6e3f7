"""CPU oracle for the 6Bit-Diffusion quantized-linear hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the C-ABI library
and its Python binding) may import or call this package; only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.

The oracle is a plain, slow, obviously-correct restatement of what the
method computes, written from the method description of "6Bit-Diffusion:
Inference-Time Mixed-Precision Quantization for Video Diffusion Models"
(technical summary, sections 2.A-2.C) and from the popular summary of the
same paper (sections 1-3), plus the public definitions of the NVFP4 / OCP
FP8 (E4M3) and E2M1 number formats.  It shares no code with the CUDA path.

Floating-point conventions: steps that the method performs in FP32
(the Hadamard butterfly, the quantizer divisions) are done here in numpy
float32, which is IEEE-754 round-to-nearest-even for every single
operation.  Reference GEMM values and statistics are computed in float64.

Module map:
  formats   small-float encoders/decoders (E2M1, E4M3, bf16, MXFP8 blocks)
  hadamard  block Fast Walsh-Hadamard transform and the dense Sylvester matrix
  quant     NVFP4 / INT8 activation quantizers, 4-bit weight packing
  gemm      reference quantized GEMMs, GELU, residual, tolerance bounds
  stats     block statistics (Gamma, cosine, max/mean outlier ratio)
  policy    per-block DMPQ / TDC / PDR decision state machine
  dit       the residual-MLP DiT chain (x + W_d GELU(W_u x) per block) under
            the policy, with a bf16 or MXFP8 delta cache

Parity status: every function here is pinned by tests in
tests/test_oracle_*.py except the policy thresholds themselves, whose
values are configuration, not something the pages fix ("parity unpinned"
for the numeric thresholds only; the decision rules are pinned by
hand-traced examples).
"""
