// Narrow-tile CTA-pair instantiations: a 256 x 128 output tile per CTA pair
// (tcgen05 cta_group::2), one CTA per SM, with a four-stage ring of two
// k-blocks per stage.
#include "gemm_inst.cuh"

namespace pts {

KernelOps kernel_ops_narrow_cg2(int kind)
{
    switch (kind) {
    case 0: return Inst<0, 2, kTileNNarrow>::ops();
    case 1: return Inst<1, 2, kTileNNarrow>::ops();
    default: return Inst<2, 2, kTileNNarrow>::ops();
    }
}

}  // namespace pts
