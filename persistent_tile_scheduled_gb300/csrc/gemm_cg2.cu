// 2-SM instantiations: a 256 x 256 output tile per CTA pair (tcgen05
// cta_group::2, cluster of 2 CTAs; each CTA loads its own halves of A and B).
#include "gemm_inst.cuh"

namespace pts {

KernelOps kernel_ops_cg2(int kind, bool full)
{
    switch (kind) {
    case 0: return full ? Inst<0, 2, kTileN, true>::ops() : Inst<0, 2, kTileN, false>::ops();
    case 1: return full ? Inst<1, 2, kTileN, true>::ops() : Inst<1, 2, kTileN, false>::ops();
    default: return full ? Inst<2, 2, kTileN, true>::ops() : Inst<2, 2, kTileN, false>::ops();
    }
}

}  // namespace pts
