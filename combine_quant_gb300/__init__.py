"""combine_quant_gb300: GB300-native MoE dispatch / combine with
pre-communication quantisation (CUDA kernels for sm_103a behind a C ABI)."""
