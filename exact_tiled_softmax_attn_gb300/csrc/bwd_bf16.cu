// placeholder, replaced by the tcgen05 backward
#include "launch.h"
namespace attn {
cudaError_t launch_bwd_bf16(const LaunchBwd&) { return cudaErrorNotSupported; }
}
