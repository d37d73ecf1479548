// k_rowgroup_f32.cu -- the f32 instances of the lanes-per-row kernel.
#include "k_rowgroup.cuh"

namespace osd {

int launch_rowgroup_f32(const Launch &l) { return rowgroup_launch_dt<kF32>(l); }

}  // namespace osd
