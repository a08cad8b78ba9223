"""GB300-native MoonEP layer path: plan, prefetch, permute, grouped GEMM,
combine and reduce_grad as sm_103a CUDA kernels behind a C ABI."""
