// The tiling query of the implicit-im2col convolution (bt_conv2d_plan_info):
// the planner's result for a geometry, read on the host without a launch.
#include "tc_conv_kernel.cuh"

namespace bt {

// defined with the planner (tc_conv.cu)
extern thread_local const ConvChoice *t_conv_force;
namespace conv {
bool choose_plan(const ConvGeom &g, bt_code code, int sms, int out_elem, ConvPlan &p);
}  // namespace conv

using namespace conv;

bool conv_plan_query(const ConvGeom &g, bt_code code, int out_elem, int sms, int pair, int split,
                     bt_conv_plan_info &info) {
    info = bt_conv_plan_info{};
    if (!conv_implicit_applies(g, code)) return false;
    const ConvChoice f{pair, 0, 0, 0, split};
    const ConvChoice *saved = t_conv_force;
    t_conv_force = &f;
    ConvPlan p;
    const bool ok = choose_plan(g, code, sms, out_elem, p);
    t_conv_force = saved;
    if (!ok) return false;
    const ConvArgs &a = p.a;
    int max_shift = 0;
    for (int t = 0; t < a.ntap; ++t) {
        const int off = static_cast<int>(a.tap[t] & 0xFFFFFu);
        if (off > max_shift) max_shift = off;
    }
    info.implicit = 1;
    info.pair = p.cp ? 1 : 0;
    info.weights_resident = a.a_resident;
    info.pixel_stages = a.b_stages;
    info.bands = a.bands;
    info.band_rows = a.ht;
    info.cta_rows = a.ht2;
    info.row_width = a.wv;
    info.tile_n = a.bn;
    info.cta_n = a.nb;
    info.staged_rows = a.rv;
    info.phases = a.nph;
    info.max_tap_shift = max_shift;
    info.tiles = a.num_tiles;
    info.smem_bytes = p.smem;
    return true;
}

}  // namespace bt
