// Narrow-tile instantiations: a 128 x 128 output tile per CTA (tcgen05
// cta_group::1), small enough in shared memory and TMEM for two CTAs per SM.
#include "gemm_inst.cuh"

namespace pts {

KernelOps kernel_ops_narrow(int kind)
{
    switch (kind) {
    case 0: return Inst<0, 1, kTileNNarrow>::ops();
    case 1: return Inst<1, 1, kTileNNarrow>::ops();
    default: return Inst<2, 1, kTileNNarrow>::ops();
    }
}

}  // namespace pts
