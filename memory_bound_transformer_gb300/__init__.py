"""GB300-native decode step of a dense Llama-style decoder.

The compute path is libmbt.so (CUDA kernels for sm_103a behind the C ABI in
include/mbt.h); this package holds its ctypes binding (capi), the weight/config
blob writer (blob), a small session wrapper (engine), the byte/FLOP ledger used
for roofline reporting (ledger) and the build step (build)."""
__all__ = ["capi", "blob", "engine", "ledger", "build"]
