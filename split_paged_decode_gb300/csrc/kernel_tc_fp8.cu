// kernel_tc_fp8.cu -- the fp8 (OCP E4M3) cache instantiations of the tcgen05
// GQA decode kernel (kernel_tc.cuh) and their geometry. The ring holds 16 KB
// E4M3 tile slots: 6 in the shallow ring (as many bytes in flight as the bf16
// kernel's three 32 KB slots), 11 in the deep ring.
#include "kernel_tc.cuh"

namespace fad {

bool tc_fp8_geometry(int qk, int ov, int rows, int nslot, bool stream_k, KernelGeometry* g)
{
    if (stream_k && nslot <= kTcSlotsShared) return false;
    if (qk != 128 || ov != 128 || rows < 1 || rows > 16) return false;
    const int nrv = rows <= 4 ? 4 : (rows <= 8 ? 8 : 16);
#define FAD_TC(NS, NRV, SLOTS)                                                                       \
    if (nslot == NS && nrv == NRV) {                                                                 \
        tc_variant<NS, NRV, true>(stream_k,                                                          \
                                  stream_k ? "tc_e4m3_d128_bn128_n16_r" #NRV "_slots" #SLOTS "_streamk" \
                                           : "tc_e4m3_d128_bn128_n16_r" #NRV "_slots" #SLOTS, g);       \
        return true;                                                                                 \
    }
    FAD_TC(3, 4, 6)
    FAD_TC(3, 8, 6)
    FAD_TC(3, 16, 6)
    FAD_TC(6, 4, 11)
    FAD_TC(6, 8, 11)
    FAD_TC(6, 16, 11)
#undef FAD_TC
    return false;
}

}  // namespace fad
