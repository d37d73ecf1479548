// k_norm_f32.cu -- the f32 instances of the LayerNorm / RMSNorm kernels.
#include "k_norm.cuh"

namespace osd {

int launch_norm_f32(const NormLaunch &l) { return norm_detail::launch_dt<kF32>(l); }

}  // namespace osd
