// k_rowgroup_bf16.cu -- the bf16 instances of the lanes-per-row kernel.
#include "k_rowgroup.cuh"

namespace osd {

int launch_rowgroup_bf16(const Launch &l) { return rowgroup_launch_dt<kBF16>(l); }

}  // namespace osd
