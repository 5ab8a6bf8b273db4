// The variants of the tcgen05 implicit-GEMM kernel that widen int8 operands
// in the kernel (normal layout with N <= 128, resident weights, no output
// options): a
// translation unit of its own so that it compiles in parallel with the others.
#include "k_igemm_kernel.cuh"

namespace {

template <int BN, int BK>
void *cvt_ptr(bool flat, bool halo) {
    if (flat)
        return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, true, false, false, false, false, false, true>);
    if (halo)
        return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, false, false, false, false, true, false, true>);
    return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, false, false, false, false, false, false, true>);
}

template <int BN>
void *cvt_bk(int bk, bool flat, bool halo) {
    switch (bk) {
    case 64: return cvt_ptr<BN, 64>(flat, halo);
    case 32: return cvt_ptr<BN, 32>(flat, halo);
    default: return cvt_ptr<BN, 16>(flat, halo);
    }
}

}  // namespace

void *igemm_select_cvt(int bn, int bk, bool flat, bool halo) {
    return bn == 128 ? cvt_bk<128>(bk, flat, halo) : cvt_bk<64>(bk, flat, halo);
}
