// kernel_tc.cu -- the bf16-cache instantiations of the tcgen05 GQA decode
// kernel (kernel_tc.cuh) and their geometry.
#include "kernel_tc.cuh"

namespace fad {

bool tc_geometry(int qk, int ov, int rows, int nslot, bool stream_k, KernelGeometry* g)
{
    if (stream_k && nslot <= kTcSlotsShared) return false;
    if (qk != 128 || ov != 128 || rows < 1 || rows > 16) return false;
    const int nrv = rows <= 4 ? 4 : (rows <= 8 ? 8 : 16);
#define FAD_TC(NS, NRV)                                                                              \
    if (nslot == NS && nrv == NRV) {                                                                 \
        tc_variant<NS, NRV, false>(stream_k,                                                         \
                                   stream_k ? "tc_d128_bn128_n16_r" #NRV "_slots" #NS "_streamk"     \
                                            : "tc_d128_bn128_n16_r" #NRV "_slots" #NS, g);           \
        return true;                                                                                 \
    }
    FAD_TC(3, 4)
    FAD_TC(3, 8)
    FAD_TC(3, 16)
    FAD_TC(6, 4)
    FAD_TC(6, 8)
    FAD_TC(6, 16)
#undef FAD_TC
    return false;
}

}  // namespace fad
