// k_norm_f16.cu -- the f16 instances of the LayerNorm / RMSNorm kernels.
#include "k_norm.cuh"

namespace osd {

int launch_norm_f16(const NormLaunch &l) { return norm_detail::launch_dt<kF16>(l); }

}  // namespace osd
