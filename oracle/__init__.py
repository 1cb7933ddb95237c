"""CPU oracle for the GPTQ layer solver (test infrastructure only).

Imported by the tests, by the package's smoke check and by the benchmark's
CPU-baseline leg; never by the product path.
"""
from .gptq_oracle import *  # noqa: F401,F403
from .gptq_oracle import (OracleConfig, LayerResult, as_config, hessian_sum,  # noqa: F401
                          hessian_entry, hessian_sum_chunked, hessian_diag,
                          hessian_columns, damped_hessian, act_order, act_order_diag, hinv_upper,
                          hinv_upper_reverse, prepare, quant_params, quantize_codes,
                          dequantize_codes, column_loop, group_index, quantize_layer,
                          rtn, dequantize, dequantize_as, dequant_matmul, round_bf16, recon_error, pack_qweight, unpack_qweight,
                          pack_qzeros, unpack_qzeros, packed_bytes, maxq_of)
