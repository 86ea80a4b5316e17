"""CPU oracle for the group-wise weight-only quantized decode GEMV/GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
product (the ``uq`` C-ABI library and its Python binding) never imports, calls or
links anything here, and nothing here imports the product: the two share no code.

What it is: a plain, slow, obviously correct restatement, in NumPy float64, of
what the decode path computes, following the "Ultra LLM Engine" page:

* section "Quantization" (table rows ``int`` and ``nf4``): group-wise uniform
  INT-N weight quantization with per-group scales, and a NormalFloat4 codebook
  quantizer; both pack low-bit codes and expose matching dequantization;
* section "Fused Kernels": the dequantized-weight GEMV (single-token decode)
  and GEMM (batched decode), i.e. y = x . W_hat^T.

The pages give no formulas; the concrete ones (symmetric INT4 scale absmax/7,
symmetric INT8 scale absmax/127, asymmetric scale (max-min)/(2^b-1) with integer
zero point, NF4 absmax times a 16-entry normal-quantile codebook, and the
two-level 256/32 super-block INT4 format w = d*sc*q - dmin*m) come from the
workload definitions this library is measured on.  Every point the definitions
leave open is resolved by the plainest reading, written at the function that
makes it.

Modules:
  fp16     -- fp16 rounding (nearest-even and toward +inf) from float64
  quant    -- quantizers and dequantizers for the six formats
  nf4      -- construction of the NF4 codebook from normal quantiles
  gemm     -- dequantize-then-matmul in float64, the error bound, the pass rule
  mlp      -- the gated MLP's fused gate/up projection silu(x W_gate^T) * (x W_up^T), its pass rule
  rope     -- RMSNorm followed by rotate-half RoPE over head_dim blocks, its pass rule
  gguf     -- decoding of GGUF Q4_0 / Q8_0 blocks (the block formats equal INT4_SYM / INT8_SYM, group 32)
  w4a8     -- dynamic per-row int8 activations and integer group sums (W4A8 / W8A8), its pass rule

Parity status: every function is pinned by ``tests/test_oracle_*.py`` against
brute force, exact rational arithmetic (``fractions.Fraction``), hand-worked
examples, closed forms and library routines, except the NF4 codebook VALUES
against any third-party table: they are this library's own construction and
are passed to both sides as an input ("parity unpinned" for that table only;
the quantile construction itself is pinned against scipy.stats.norm.ppf).
"""
