// The variants of the tcgen05 implicit-GEMM kernel for layers with output
// options (a residual, upsample replicas): a translation unit of its own so
// that both halves of the family compile in parallel.
#include "k_igemm_kernel.cuh"

namespace {

template <int BN, int BK, bool FLAT, bool SWAP, bool PAIR>
void *fused_ptr() {
    return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, FLAT, SWAP, PAIR, true>);
}

template <int BN, int BK, bool SWAP, bool PAIR>
void *fused_flat(bool flat) {
    return flat ? fused_ptr<BN, BK, true, SWAP, PAIR>() : fused_ptr<BN, BK, false, SWAP, PAIR>();
}

template <int BN, bool SWAP, bool PAIR>
void *fused_bk(int bk, bool flat) {
    switch (bk) {
    case 64: return fused_flat<BN, 64, SWAP, PAIR>(flat);
    case 32: return fused_flat<BN, 32, SWAP, PAIR>(flat);
    default: return fused_flat<BN, 16, SWAP, PAIR>(flat);
    }
}

}  // namespace

void *igemm_select_fused(int bn, int bk, bool flat, bool swap, bool pair) {
    if (pair) return bn == 128 ? fused_bk<128, false, true>(bk, flat) : fused_bk<256, false, true>(bk, flat);
    if (swap) return fused_bk<128, true, false>(bk, flat);
    switch (bn) {
    case 256: return fused_bk<256, false, false>(bk, flat);
    case 128: return fused_bk<128, false, false>(bk, flat);
    default: return fused_bk<64, false, false>(bk, flat);
    }
}
