"""CPU oracle for the W2A8 ternary linear -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline and
``--impl reference`` legs may import this package; the CUDA library and its
binding never do."""
from .w2a8 import (  # noqa: F401
    QMAX, TILE_N, TILE_K, TILE_BYTES, TRAILER_MAGIC,
    bf16_bits_to_f32, f32_to_bf16_bits, ternarize_absmean, quant_act,
    quant_act_bf16, gemm_acc, dequant, w2a8_linear, dequant_chain, linear_chain, packed_bytes,
    FP8_MAX, e4m3_round, quant_act_fp8, quant_act_fp8_bf16, gemm_acc_fp8, fp8_linear, pack_tiles,
    unpack_tiles, read_trailer,
)
