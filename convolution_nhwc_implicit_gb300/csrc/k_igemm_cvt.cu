// The variants of the tcgen05 implicit-GEMM kernel with a converter
// warpgroup (normal layout with N <= 128, resident weights, no output
// options): int8 operands widened in the kernel, and the k_w-folded
// small-channel bf16 stem assembled in the kernel.  A translation unit of
// its own so that it compiles in parallel with the others.
#include "k_igemm_kernel.cuh"

namespace {

template <int BN, int BK, bool EPT>
void *widen_ptr(bool flat, bool halo) {
    if (flat)
        return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, true, false, false, false, false, EPT, 1>);
    if (halo)
        return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, false, false, false, false, true, EPT, 1>);
    return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, false, false, false, false, false, EPT, 1>);
}

template <int BN>
void *widen_bk(int bk, bool flat, bool halo, bool ept) {
    switch (bk) {
    case 64: return ept ? widen_ptr<BN, 64, true>(flat, halo) : widen_ptr<BN, 64, false>(flat, halo);
    case 32: return ept ? widen_ptr<BN, 32, true>(flat, halo) : widen_ptr<BN, 32, false>(flat, halo);
    default: return ept ? widen_ptr<BN, 16, true>(flat, halo) : widen_ptr<BN, 16, false>(flat, halo);
    }
}

// (the folded operand is one 16-channel K block per filter row: BK = 16, spatial)
template <int BN>
void *fold_ptr(bool halo, bool ept) {
    if (halo)
        return ept ? reinterpret_cast<void *>(&igemm_bf16_kernel<BN, 16, false, false, false, false, true, true, 2>)
                   : reinterpret_cast<void *>(&igemm_bf16_kernel<BN, 16, false, false, false, false, true, false, 2>);
    return ept ? reinterpret_cast<void *>(&igemm_bf16_kernel<BN, 16, false, false, false, false, false, true, 2>)
               : reinterpret_cast<void *>(&igemm_bf16_kernel<BN, 16, false, false, false, false, false, false, 2>);
}

}  // namespace

void *igemm_select_cvt(int mode, int bn, int bk, bool flat, bool halo, bool ept, int mb) {
    if (mode == 2 && mb == 2)  // (two M blocks a tile: N = 64, halo staging, an epilogue per tile)
        return bn == 64 && halo && ept
                   ? reinterpret_cast<void *>(&igemm_bf16_kernel<64, 16, false, false, false, false, true, true, 2, 2>)
                   : nullptr;
    if (mode == 2) return bn == 128 ? fold_ptr<128>(halo, ept) : fold_ptr<64>(halo, ept);
    return bn == 128 ? widen_bk<128>(bk, flat, halo, ept) : widen_bk<64>(bk, flat, halo, ept);
}
