// 2-SM instantiations: a 256 x 256 output tile per CTA pair (tcgen05
// cta_group::2, cluster of 2 CTAs; each CTA loads its own halves of A and B).
#include "gemm_inst.cuh"

namespace pts {

KernelOps kernel_ops_cg2(int kind)
{
    switch (kind) {
    case 0: return Inst<0, 2>::ops();
    case 1: return Inst<1, 2>::ops();
    default: return Inst<2, 2>::ops();
    }
}

}  // namespace pts
