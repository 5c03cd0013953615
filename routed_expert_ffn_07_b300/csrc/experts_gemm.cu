// Prefill experts (grouped tensor-core GEMM): placeholder until the tcgen05 path lands.
#include "common.cuh"
namespace moe {
cudaError_t gemm_kernels_init(int) { return cudaSuccess; }
size_t gemm_workspace_bytes(int, int, int, int, int) { return 256; }
cudaError_t launch_experts_gemm(const ExpertArgs&, void*, cudaStream_t, cudaEvent_t) { return cudaErrorNotSupported; }
}  // namespace moe
