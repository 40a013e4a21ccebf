"""GB300-native FP16 linear: y = FP16(x . W^T) + b on sm_103a.

``linear(x, w, b)`` is the tensor-level call, and ``contract`` the widened
contraction (bfloat16 heads, no bias, FP32 output, fused epilogue steps);
``column_parallel_linear`` and ``row_parallel_linear`` split the op over
torch.distributed ranks;
the C entry points of include/poot_linear.h are mirrored one to one in
``binding``.
"""
from .binding import (  # noqa: F401
    GEMV_MAX_M, Options, options, POOT_ERR_CUDA, POOT_ERR_DEVICE_TIMEOUT, POOT_ERR_INVALID_ARG,
    POOT_ERR_MISALIGNED, POOT_ERR_UNSUPPORTED_DEVICE, POOT_OK, PootLinearError,
    VARIANT_AUTO, VARIANT_BIAS_ONLY, VARIANT_GEMM_CPASYNC, VARIANT_GEMM_REG,
    VARIANT_GEMM_TMA, VARIANT_GEMM_PACKED, VARIANT_GEMV, VARIANT_GEMV_SCALAR, VARIANT_NAMES, VARIANT_NONE,
    library_path, linear, load_library, poot_linear, poot_linear_device_status, poot_linear_f16,
    poot_linear_f16_ex, poot_linear_f16_variant, poot_linear_last_cuda_error,
    poot_linear_status_string, poot_linear_version, variant_for,
    ContractionSpec, DTYPE_BF16, DTYPE_F16, EP_ADD, EP_GELU_ERF, EP_GELU_TANH, EP_MUL, EP_SILU,
    EPILOGUE_MAX_STEPS, EpilogueStep, contract, poot_contract, poot_contract_grouped,
    NOALLOC_SCRATCH_BYTES, poot_linear_f16_splitk_noalloc,
    poot_linear_tp_shard, poot_linear_gather_columns, poot_linear_f16_finish, poot_linear_gemm_plan,
)
from .tensor_parallel import (  # noqa: F401
    shard_range, column_parallel_linear, row_parallel_linear,
)

__version__ = "0.1.0"
