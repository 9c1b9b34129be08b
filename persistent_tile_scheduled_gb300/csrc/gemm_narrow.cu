// Narrow-tile instantiations: a 128 x 128 output tile per CTA (tcgen05
// cta_group::1), small enough in shared memory and TMEM for two CTAs per SM.
#include "gemm_inst.cuh"

namespace pts {

KernelOps kernel_ops_narrow(int kind, bool full)
{
    switch (kind) {
    case 0: return full ? Inst<0, 1, kTileNNarrow, true>::ops() : Inst<0, 1, kTileNNarrow, false>::ops();
    case 1: return full ? Inst<1, 1, kTileNNarrow, true>::ops() : Inst<1, 1, kTileNNarrow, false>::ops();
    default: return full ? Inst<2, 1, kTileNNarrow, true>::ops() : Inst<2, 1, kTileNNarrow, false>::ops();
    }
}

}  // namespace pts
