// k_rowgroup_f16.cu -- the f16 instances of the lanes-per-row kernel.
#include "k_rowgroup.cuh"

namespace osd {

int launch_rowgroup_f16(const Launch &l) { return rowgroup_launch_dt<kF16>(l); }

}  // namespace osd
