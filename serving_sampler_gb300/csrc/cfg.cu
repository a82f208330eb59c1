// placeholder until the CFG kernels land
#include "sv_internal.h"
namespace sv {
size_t cfg_workspace_bytes(int64_t, int32_t, int32_t, int32_t) { return 256; }
cudaError_t launch_cfg_merge_sample(const Rows&, const Rows&, const CfgShape&, const Rows*, int32_t,
                                    int32_t, const int32_t*, const uint64_t*, const float*, int32_t*,
                                    int32_t*, float*, int32_t*, void*, cudaStream_t)
{
    return cudaErrorNotSupported;
}
}  // namespace sv
