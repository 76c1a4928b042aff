// placeholder until the tcgen05 grouped GEMM lands
#include "common.cuh"
#include "internal.h"
namespace moe {
bool tc_available() { return false; }
size_t tc_grouped_ws_bytes(int) { return 0; }
cudaError_t launch_tc_grouped_swiglu_fwd(const Ctx&, int, int64_t, int, int, const int32_t*,
                                         const void*, const void*, const void*, void*, void*,
                                         void*, void*, int*) { return cudaErrorNotSupported; }
cudaError_t launch_tc_grouped_swiglu_bwd(const Ctx&, int, int64_t, int, int, const int32_t*,
                                         const void*, const void*, const void*, const void*,
                                         const void*, const void*, void*, void*, void*, void*,
                                         void*, int*) { return cudaErrorNotSupported; }
}
