"""CPU oracle for the AWQ W4A16 GEMM-layout linear (test infrastructure only;
see awq_oracle.py)."""
from .awq_oracle import (ORDER, REVERSE_ORDER, resolve_group_size, unpack_codes,
                         pack_codes, dequant_f32, dequant_f16, dequant_page_layout,
                         gemm, gemm_sampled, gemm_rows, dequant_columns_f32,
                         within_tolerance, quantize_rtn, round_to_bf16, dequant_bf16,
                         gemm_grouped, unpack_codes8, pack_codes8, dequant8_f32, gemm8,
                         repack, repack_size, unpack_repacked, gemm_packed,
                         repack8, repack8_size, unpack_repacked8, gemm_packed8)

__all__ = ["ORDER", "REVERSE_ORDER", "resolve_group_size", "unpack_codes", "pack_codes",
           "dequant_f32", "dequant_f16", "dequant_page_layout", "gemm", "gemm_sampled",
           "gemm_rows", "dequant_columns_f32", "within_tolerance", "quantize_rtn",
           "round_to_bf16", "dequant_bf16", "gemm_grouped",
           "unpack_codes8", "pack_codes8", "dequant8_f32", "gemm8",
           "repack", "repack_size", "unpack_repacked", "gemm_packed",
           "repack8", "repack8_size", "unpack_repacked8", "gemm_packed8"]
