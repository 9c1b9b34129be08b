// Narrow-tile CTA-pair instantiations: a 256 x 128 output tile per CTA pair
// (tcgen05 cta_group::2), one CTA per SM, with a four-stage ring of two
// k-blocks per stage.
#include "gemm_inst.cuh"

namespace pts {

KernelOps kernel_ops_narrow_cg2(int kind, bool full)
{
    switch (kind) {
    case 0: return full ? Inst<0, 2, kTileNNarrow, true>::ops() : Inst<0, 2, kTileNNarrow, false>::ops();
    case 1: return full ? Inst<1, 2, kTileNNarrow, true>::ops() : Inst<1, 2, kTileNNarrow, false>::ops();
    default: return full ? Inst<2, 2, kTileNNarrow, true>::ops() : Inst<2, 2, kTileNNarrow, false>::ops();
    }
}

}  // namespace pts
