// k_norm_bf16.cu -- the bf16 instances of the LayerNorm / RMSNorm kernels.
#include "k_norm.cuh"

namespace osd {

int launch_norm_bf16(const NormLaunch &l) { return norm_detail::launch_dt<kBF16>(l); }

}  // namespace osd
