"""Weight-only quantized linear layers (MLX affine 4/6/8-bit, group 64) for GB300.

The CUDA library and its binding live in ``weight_only_bit_mlx_gb300.qlinear``; the
seeded input generators in ``weight_only_bit_mlx_gb300.synth``.  Importing this
package does not load the CUDA library.
"""
