"""GB300-native parallel Newton forward of a diagonal-mix GRU.

The computation runs in ``libnrnn.so`` (hand-written CUDA for sm_103a, C ABI in
``include/nrnn.h``); this package is its Python binding.  Importing it loads
the library and fails if it cannot."""
from ._binding import (  # noqa: F401
    ALGOS,
    EXPORTED,
    GATE_ORDER,
    AgreementError,
    AgreementReport,
    DeviceCuSeqlens,
    NewtonDivergenceError,
    NrnnError,
    bounded_wait,
    debug_withhold_publish,
    decode_step,
    default_agreement_atol,
    head_mask,
    host_staging_bytes,
    input_projection,
    lib_path,
    load,
    lookback_form,
    newton_backward,
    newton_forward,
    newton_forward_host,
    newton_forward_x,
    newton_forward_x_host,
    pack_plan,
    params_tensor,
    picard,
    probe_xu_rates,
    projection_workspace_bytes,
    residual,
    sequential_forward,
    set_wait_limit_ns,
    validate_cu_seqlens,
    verify_agreement,
    workspace_bytes,
    x_host_staging_bytes,
)

load()
