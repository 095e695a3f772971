// Host side of the implicit-im2col binary convolution (kernel in
// tc_conv_kernel.cuh): the plan of a geometry (tiles, phase images, taps,
// shared-memory layout), the tensor maps, and the launches.
#include <atomic>
#include <utility>
#include <vector>

#include "tc_conv_kernel.cuh"

namespace bt {

// The calling thread's forced plan (bt_tune_conv2d, or a kept winner for the
// call in progress).
thread_local const ConvChoice *t_conv_force = nullptr;

namespace conv {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

uint32_t make_idesc(int code, int m, int bn) {
    const uint32_t mn = ((static_cast<uint32_t>(bn) >> 3) << 17) | ((static_cast<uint32_t>(m) >> 4) << 24);
    if (code == BT_CODE_E4M3) return (1u << 4) | mn;                             // E4M3 x E4M3 -> F32
    return (1u << 7) | (1u << 10) | (1u << 23) | mn;   // block-scaled E2M1 x E2M1, UE8M0 scales, ids 0
}

int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }


// The implicit plan of a convolution, or false where it does not apply (the
// caller then unfolds explicitly): E2M1 / E4M3 codes, stride 1 or 2, at most
// 64 taps, a virtual row that fits one tile, copies within TMA's box limits,
// and shared memory for the weights (resident or a ring of at least two
// stages) beside two pixel stages and the epilogue's staging.
bool plan_conv(const ConvGeom &g, bt_code code, int sms, int out_elem, ConvPlan &p, bool cp = false) {
    if (code != BT_CODE_E2M1 && code != BT_CODE_E4M3) return false;
    if (g.s < 1 || g.s > 2 || g.k < 1 || g.k * g.k > kMaxTaps) return false;
    if (g.B < 1 || g.B > (int64_t(1) << 24) || g.O < 1 || g.O > (int64_t(1) << 24)) return false;
    if (g.Ho < 1 || g.Wo < 1 || g.Ho > 65536 || g.Wo > 256 || g.H > (int64_t(1) << 30) || g.W > (int64_t(1) << 30))
        return false;
    const int64_t cb = row_bytes(g.C, code);
    const int sw = cb % 128 == 0 ? 128 : 64;
    if (cb % sw != 0) return false;
    ConvArgs &a = p.a;
    std::memset(&a, 0, sizeof(a));
    a.B = static_cast<int>(g.B);
    a.O = static_cast<int>(g.O);
    a.Ho = static_cast<int>(g.Ho);
    a.Wo = static_cast<int>(g.Wo);
    a.sw = sw;
    a.nsl = static_cast<int>(cb / sw);
    a.ntap = g.k * g.k;
    a.stride = g.s;
    if (static_cast<int64_t>(a.ntap) * a.nsl > 65535) return false;
    // phases and tap offsets (along one axis: e = -p + kk*d = s*q + ph)
    const int s = g.s;
    int phase_id[4] = {-1, -1, -1, -1};
    int qy_min[4], qx_min[4], qx_span = 0;
    int nph = 0;
    for (int kh = 0; kh < g.k; ++kh)
        for (int kw = 0; kw < g.k; ++kw) {
            const int ey = -g.p + kh * g.d, ex = -g.p + kw * g.d;
            const int qy = floor_div(ey, s), qx = floor_div(ex, s);
            const int key = (ey - s * qy) * 2 + (ex - s * qx);
            if (phase_id[key] < 0) {
                phase_id[key] = nph;
                qy_min[nph] = qy;
                qx_min[nph] = qx;
                a.ph_y0[nph] = s * qy + (ey - s * qy);
                a.ph_x0[nph] = s * qx + (ex - s * qx);
                ++nph;
            }
            const int id = phase_id[key];
            if (qy < qy_min[id]) { qy_min[id] = qy; a.ph_y0[id] = s * qy + (ey - s * qy); }
            if (qx < qx_min[id]) { qx_min[id] = qx; a.ph_x0[id] = s * qx + (ex - s * qx); }
        }
    a.nph = nph;
    int qy_off_max = 0, qx_off_max = 0;
    for (int kh = 0; kh < g.k; ++kh)
        for (int kw = 0; kw < g.k; ++kw) {
            const int ey = -g.p + kh * g.d, ex = -g.p + kw * g.d;
            const int qy = floor_div(ey, s), qx = floor_div(ex, s);
            const int id = phase_id[(ey - s * qy) * 2 + (ex - s * qx)];
            if (qy - qy_min[id] > qy_off_max) qy_off_max = qy - qy_min[id];
            if (qx - qx_min[id] > qx_off_max) qx_off_max = qx - qx_min[id];
        }
    qx_span = qx_off_max;
    a.wv = a.Wo + qx_span;
    const int bn_max = code == BT_CODE_E2M1 ? 240 : 256;
    // an even row width keeps pixel pairs of an even Wo aligned in the output
    if (a.Wo % 2 == 0 && a.wv % 2 == 1 && a.wv + 1 <= bn_max) a.wv += 1;
    if (a.wv > bn_max || a.wv * s > 256) return false;
    p.cp = cp;
    // BT_CONV_SPLIT=n (or a forced plan's split) cuts each image into n times
    // as many bands as fit a tile: more, narrower tiles
    int split = 1;
    if (const char *env = std::getenv("BT_CONV_SPLIT")) split = std::atoi(env);
    else if (t_conv_force != nullptr && t_conv_force->split > 1) split = t_conv_force->split;
    if (split < 1) split = 1;
    if (split > 8) split = 8;
    if (!cp) {
        int ht = bn_max / a.wv;
        if (ht > a.Ho) ht = a.Ho;
        a.bands = (a.Ho + ht - 1) / ht;
        if (split > 1) a.bands = a.bands * split < a.Ho ? a.bands * split : a.Ho;
        a.ht = (a.Ho + a.bands - 1) / a.bands;       // balance the bands
        a.bands = (a.Ho + a.ht - 1) / a.ht;          // (a split leaves no band empty)
        a.bn = (a.ht * a.wv + 15) / 16 * 16;
        if (a.bn < 32) a.bn = 32;
        if (a.bn > bn_max) return false;
        a.ht2 = a.ht;
        a.nb = a.bn;
    } else {
        // a pair: ht2 rows per CTA, each CTA's nb columns a multiple of 8
        int ht2 = (bn_max / 2) / a.wv;
        if (ht2 > (a.Ho + 1) / 2) ht2 = (a.Ho + 1) / 2;
        if (ht2 < 1) return false;
        a.bands = (a.Ho + 2 * ht2 - 1) / (2 * ht2);
        if (split > 1) a.bands = a.bands * split < (a.Ho + 1) / 2 ? a.bands * split : (a.Ho + 1) / 2;
        a.ht2 = (a.Ho + 2 * a.bands - 1) / (2 * a.bands);   // balance the bands
        a.bands = (a.Ho + 2 * a.ht2 - 1) / (2 * a.ht2);      // (a split leaves no band empty)
        a.ht = 2 * a.ht2;
        a.nb = (a.ht2 * a.wv + 7) / 8 * 8;
        if (a.nb < 16) a.nb = 16;
        a.bn = 2 * a.nb;
        if (a.bn > bn_max) return false;
    }
    int max_off = 0;
    for (int kh = 0; kh < g.k; ++kh)
        for (int kw = 0; kw < g.k; ++kw) {
            const int ey = -g.p + kh * g.d, ex = -g.p + kw * g.d;
            const int qy = floor_div(ey, s), qx = floor_div(ex, s);
            const int id = phase_id[(ey - s * qy) * 2 + (ex - s * qx)];
            const int off = (qy - qy_min[id]) * a.wv + (qx - qx_min[id]);
            a.tap[kh * g.k + kw] = (static_cast<uint32_t>(kh * g.k + kw) << 24) | (static_cast<uint32_t>(id) << 20) |
                                   static_cast<uint32_t>(off);
            if (off > max_off) max_off = off;
        }
    a.rv = (a.nb + max_off + a.wv - 1) / a.wv;       // rows staged per CTA
    if (a.rv * s > 256) return false;
    a.img_tx = static_cast<uint32_t>(a.rv * a.wv * sw);
    a.img_bytes = (a.img_tx + 1023u) / 1024u * 1024u;
    a.stage_bytes = static_cast<uint32_t>(a.nph * a.nsl) * a.img_bytes;
    a.num_ot = (a.O + (cp ? 2 : 1) * kBM - 1) / ((cp ? 2 : 1) * kBM);
    const int64_t tiles = static_cast<int64_t>(a.num_ot) * a.B * a.bands;
    if (tiles > (int64_t(1) << 30)) return false;
    a.num_tiles = static_cast<int>(tiles);
    // weights resident (loaded once per CTA, each CTA keeping one channel
    // tile) or streamed through a ring of slices re-read per tile; one or two
    // pixel stages. Preference: resident + two stages; resident + one stage
    // when a CTA gets at most two tiles (only the second tile's copy is then
    // exposed); streamed + two stages; resident + one; streamed + one.
    // BT_CONV_PLAN=r2|r1|s2|s1 picks one where it fits.
    const int nslices = a.ntap * a.nsl;
    const int64_t slice_a = static_cast<int64_t>(kBM) * sw;
    int units = cp ? sms / 2 : sms;                  // CTAs, or pairs
    if (units > a.num_tiles) units = a.num_tiles;
    int a_d_res = 1;
    for (int d = 8; d >= 1; --d)
        if (nslices % d == 0) { a_d_res = d; break; }
    const int64_t a_res_bytes = static_cast<int64_t>(nslices) * slice_a;
    auto fixed_of = [&](int bst) {
        return kReserve + staging_bytes(out_elem) + static_cast<int64_t>(bst) * a.stage_bytes;
    };
    auto fits_res = [&](int bst) { return units >= a.num_ot && fixed_of(bst) + a_res_bytes <= kSmemMax; };
    auto stream_d = [&](int bst, int *stages) {
        for (int d = 4; d >= 1; --d) {
            if (nslices % d != 0) continue;
            const int64_t room = kSmemMax - fixed_of(bst);
            const int64_t st = room > 0 ? room / (d * slice_a) : 0;
            if (st >= 2) { *stages = static_cast<int>(st > kMaxAStages ? kMaxAStages : st); return d; }
        }
        return 0;
    };
    int st2 = 0, st1 = 0;
    const int sd2 = stream_d(2, &st2), sd1 = stream_d(1, &st1);
    const bool few = a.num_tiles <= 2 * ((units / a.num_ot) * a.num_ot > 0 ? (units / a.num_ot) * a.num_ot : units);
    char plan = 0;                                   // 'R' resident, 'S' streamed
    int bst = 2;
    if (const char *env = std::getenv("BT_CONV_PLAN")) {
        if (std::strcmp(env, "r2") == 0 && fits_res(2)) { plan = 'R'; bst = 2; }
        else if (std::strcmp(env, "r1") == 0 && fits_res(1)) { plan = 'R'; bst = 1; }
        else if (std::strcmp(env, "s2") == 0 && sd2) { plan = 'S'; bst = 2; }
        else if (std::strcmp(env, "s1") == 0 && sd1) { plan = 'S'; bst = 1; }
    } else if (const ConvChoice *f = t_conv_force) {
        if (f->plan == 'R' && (f->bst == 1 || f->bst == 2) && fits_res(f->bst)) { plan = 'R'; bst = f->bst; }
        else if (f->plan == 'S' && f->bst == 2 && sd2) { plan = 'S'; bst = 2; }
        else if (f->plan == 'S' && f->bst == 1 && sd1) { plan = 'S'; bst = 1; }
    }
    if (plan == 0) {
        if (fits_res(2)) { plan = 'R'; bst = 2; }
        else if (few && fits_res(1)) { plan = 'R'; bst = 1; }
        else if (sd2) { plan = 'S'; bst = 2; }
        else if (fits_res(1)) { plan = 'R'; bst = 1; }
        else if (sd1) { plan = 'S'; bst = 1; }
        else return false;
    }
    a.b_stages = bst;
    if (plan == 'R') {
        a.a_resident = 1;
        a.a_d = a_d_res;
        a.a_boxes = nslices / a_d_res;
        a.a_stages = 0;
        units = units / a.num_ot * a.num_ot;
        p.smem = static_cast<int>(fixed_of(bst) + a_res_bytes);
    } else {
        a.a_resident = 0;
        a.a_boxes = 0;
        a.a_d = bst == 2 ? sd2 : sd1;
        a.a_stages = bst == 2 ? st2 : st1;
        p.smem = static_cast<int>(fixed_of(bst) + static_cast<int64_t>(a.a_stages) * a.a_d * slice_a);
    }
    if (p.smem > kSmemMax) return false;
    p.grid = (units < 1 ? 1 : units) * (cp ? 2 : 1);
    a.idesc = make_idesc(code, cp ? 2 * kBM : kBM, a.bn);
    a.pairs = (a.wv % 2 == 0 && a.Wo % 2 == 0 && (static_cast<int64_t>(a.Ho) * a.Wo) % 2 == 0) ? 1 : 0;
    return true;
}

// The weights' map: [O, k*k*cb] as {sw bytes, O rows, k*k*nsl slices}.
bool encode_weight_map(const ConvGeom &g, bt_code code, const ConvArgs &a, const uint8_t *wp, CUtensorMap *ma) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    const uint64_t cb = static_cast<uint64_t>(row_bytes(g.C, code));
    const CUtensorMapSwizzle swz = a.sw == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.sw), static_cast<cuuint64_t>(g.O),
                              static_cast<cuuint64_t>(a.ntap * a.nsl)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.ntap) * cb, static_cast<cuuint64_t>(a.sw)};
        cuuint32_t box[3] = {static_cast<cuuint32_t>(a.sw), static_cast<cuuint32_t>(kBM),
                             static_cast<cuuint32_t>(a.a_d)};
        cuuint32_t es[3] = {1, 1, 1};
        if (fn(ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(wp), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

// Both maps: the weights', and the packed pixels' [B, H, W, cb] as {cb bytes,
// W, H, B}, a box taking one slice of wv columns and rv rows with traversal
// stride s.
bool encode_maps(const ConvGeom &g, bt_code code, const ConvArgs &a, const uint8_t *xp, const uint8_t *wp,
                 CUtensorMap *ma, CUtensorMap *mb) {
    if (!encode_weight_map(g, code, a, wp, ma)) return false;
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    const uint64_t cb = static_cast<uint64_t>(row_bytes(g.C, code));
    const CUtensorMapSwizzle swz = a.sw == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    {
        cuuint64_t dims[4] = {cb, static_cast<cuuint64_t>(g.W), static_cast<cuuint64_t>(g.H),
                              static_cast<cuuint64_t>(g.B)};
        cuuint64_t strides[3] = {cb, static_cast<cuuint64_t>(g.W) * cb, static_cast<cuuint64_t>(g.H * g.W) * cb};
        cuuint32_t box[4] = {static_cast<cuuint32_t>(a.sw), static_cast<cuuint32_t>(a.wv * a.stride),
                             static_cast<cuuint32_t>(a.rv * a.stride), 1};
        cuuint32_t es[4] = {1, static_cast<cuuint32_t>(a.stride), static_cast<cuuint32_t>(a.stride), 1};
        if (fn(mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t *>(xp), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

// The plan a launch takes: CTA pairs (M = 256 tiles) where the layer has more
// than 128 output channels and the pair plan fits, else single CTAs.
// BT_CONV_PAIR=0 or 1 in the environment forces one or the other (1 where it
// fits).
bool choose_plan(const ConvGeom &g, bt_code code, int sms, int out_elem, ConvPlan &p) {
    int want = -1;
    if (const char *env = std::getenv("BT_CONV_PAIR")) want = std::strcmp(env, "0") == 0 ? 0 : 1;
    else if (t_conv_force != nullptr && (t_conv_force->pair == 0 || t_conv_force->pair == 1)) want = t_conv_force->pair;
    if (want != 0 && sms >= 2 && (want == 1 || g.O > kBM) && plan_conv(g, code, sms, out_elem, p, true)) return true;
    return plan_conv(g, code, sms, out_elem, p, false);
}

// The packing warps' part of the plan: which phase image each input pixel
// parity feeds, the span of the phases' first rows, and whether staged rows
// past the image must be cleared per tile (several bands per image).
void plan_fused(const ConvGeom &g, bt_code code, ConvPlan &p) {
    ConvArgs &a = p.a;
    a.C = static_cast<int>(g.C);
    a.H = static_cast<int>(g.H);
    a.W = static_cast<int>(g.W);
    a.HW = static_cast<int>(g.H * g.W);
    a.ncg = static_cast<int>(row_bytes(g.C, code) / (code == BT_CODE_E2M1 ? 16 : 32));
    a.div_w = make_fastdiv(static_cast<uint32_t>(g.W));
    for (int i = 0; i < 4; ++i) a.ph_of[i] = -1;
    a.ph_ymin = a.ph_y0[0];
    a.ph_ymax = a.ph_y0[0];
    for (int ph = 0; ph < a.nph; ++ph) {
        const int py = ((a.ph_y0[ph] % 2) + 2) % 2, px = ((a.ph_x0[ph] % 2) + 2) % 2;
        if (a.stride == 2) a.ph_of[py * 2 + px] = ph;
        if (a.ph_y0[ph] < a.ph_ymin) a.ph_ymin = a.ph_y0[ph];
        if (a.ph_y0[ph] > a.ph_ymax) a.ph_ymax = a.ph_y0[ph];
    }
    if (a.stride == 1) a.ph_of[0] = 0;
    a.zero_rows = a.bands > 1 ? 1 : 0;
    a.prefetch = 1;
    if (const char *env = std::getenv("BT_CONV_PREFETCH")) a.prefetch = std::strcmp(env, "0") != 0;
}

}  // namespace conv

using namespace conv;

// ---------------------------------------------------------------------------
// measured selection: candidates, the forced plan, the kept winners
// ---------------------------------------------------------------------------

void conv_force(const ConvChoice *c) { t_conv_force = c; }
const ConvChoice *conv_forced() { return t_conv_force; }

int conv_candidates(const ConvGeom &g, bt_code code, bt_dtype x_dtype, bt_dtype out_t, ConvChoice *out, int max) {
    const ConvChoice *saved = t_conv_force;
    t_conv_force = nullptr;
    int n = 0;
    auto add = [&](const ConvChoice &c) {
        if (n >= max) return;
        for (int i = 0; i < n; ++i)
            if (out[i].pair == c.pair && out[i].plan == c.plan && out[i].bst == c.bst && out[i].fused == c.fused &&
                (out[i].split > 1 ? out[i].split : 1) == (c.split > 1 ? c.split : 1))
                return;
        out[n++] = c;
    };
    if (max > 0 && out != nullptr && conv_implicit_applies(g, code)) {
        const int oe = out_t == BT_BF16 || out_t == BT_F16 ? 2 : 4;
        const int sms = device_sm_count();
        // the plan a launch takes under forced choice f (nullptr: the planner's
        // own), and its bands per image
        auto effective = [&](const ConvChoice *f, ConvChoice &c, int &bands) {
            t_conv_force = f;
            ConvPlan p;
            const bool ok = choose_plan(g, code, sms, oe, p);
            t_conv_force = nullptr;
            if (!ok) return false;
            c = ConvChoice{p.cp ? 1 : 0, p.a.a_resident ? 'R' : 'S', p.a.b_stages, 0, f != nullptr ? f->split : 0};
            bands = p.a.bands;
            return true;
        };
        ConvChoice c{};
        int bands = 0;
        if (effective(nullptr, c, bands)) add(c);
        const int plans[4][2] = {{'R', 2}, {'R', 1}, {'S', 2}, {'S', 1}};
        for (int pair = 1; pair >= 0; --pair)
            for (const auto &pl : plans) {
                const ConvChoice f{pair, pl[0], pl[1], 0, 0};
                int b0 = 0;
                if (!(effective(&f, c, b0) && c.pair == f.pair && c.plan == f.plan && c.bst == f.bst)) continue;
                add(c);
                // the same plan over more bands, where that changes the tiling
                int last = b0;
                for (int sp = 2; sp <= 4; sp *= 2) {
                    const ConvChoice fs{pair, pl[0], pl[1], 0, sp};
                    int bs = 0;
                    if (effective(&fs, c, bs) && c.pair == fs.pair && c.plan == fs.plan && c.bst == fs.bst &&
                        bs > last) {
                        add(c);
                        last = bs;
                    }
                }
            }
        // each plan again with the convolution packing x itself, where it can
        bool fused_ok = false;
        if (x_dtype == BT_F32 || x_dtype == BT_BF16 || x_dtype == BT_F16) {
            const ConvChoice f{-1, 0, 0, 1, 0};
            t_conv_force = &f;
            fused_ok = conv_fused_applies(g, code, x_dtype);
            t_conv_force = nullptr;
        }
        if (fused_ok) {
            const int m = n;
            for (int i = 0; i < m; ++i) {
                ConvChoice f = out[i];
                f.fused = 1;
                add(f);
            }
        }
    }
    t_conv_force = saved;
    return n;
}

namespace {
struct ConvKey {
    int dev;
    int64_t B, C, H, W, O;
    int k, s, p, d, code, out_t;
    bool same_geometry(const ConvKey &o) const {
        return dev == o.dev && B == o.B && C == o.C && H == o.H && W == o.W && k == o.k && s == o.s && p == o.p &&
               d == o.d && code == o.code;
    }
    bool operator==(const ConvKey &o) const { return same_geometry(o) && O == o.O && out_t == o.out_t; }
};
std::mutex g_conv_mu;
std::vector<std::pair<ConvKey, ConvChoice>> g_conv_kept;      // most recent last
std::atomic<int> g_conv_count{0};

ConvKey conv_key(const ConvGeom &g, bt_code code, bt_dtype out_t) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    return ConvKey{dev, g.B, g.C, g.H, g.W, g.O, g.k, g.s, g.p, g.d, static_cast<int>(code), static_cast<int>(out_t)};
}
}  // namespace

void conv_remember(const ConvGeom &g, bt_code code, bt_dtype out_t, const ConvChoice &c) {
    const ConvKey key = conv_key(g, code, out_t);
    std::lock_guard<std::mutex> lock(g_conv_mu);
    for (size_t i = 0; i < g_conv_kept.size(); ++i)
        if (g_conv_kept[i].first == key) {
            g_conv_kept.erase(g_conv_kept.begin() + static_cast<std::ptrdiff_t>(i));
            break;
        }
    g_conv_kept.emplace_back(key, c);
    g_conv_count.store(static_cast<int>(g_conv_kept.size()), std::memory_order_release);
}

bool conv_lookup(const ConvGeom &g, bt_code code, bt_dtype out_t, ConvChoice &c) {
    if (g_conv_count.load(std::memory_order_acquire) == 0) return false;
    const ConvKey key = conv_key(g, code, out_t);
    std::lock_guard<std::mutex> lock(g_conv_mu);
    for (const auto &e : g_conv_kept)
        if (e.first == key) {
            c = e.second;
            return true;
        }
    return false;
}

bool conv_kept_fused(const ConvGeom &g, bt_code code, bool &fused) {
    if (g_conv_count.load(std::memory_order_acquire) == 0) return false;
    const ConvKey key = conv_key(g, code, BT_F32);
    std::lock_guard<std::mutex> lock(g_conv_mu);
    for (auto it = g_conv_kept.rbegin(); it != g_conv_kept.rend(); ++it)
        if (it->first.same_geometry(key)) {
            fused = it->second.fused == 1;
            return true;
        }
    return false;
}

void conv_forget() {
    std::lock_guard<std::mutex> lock(g_conv_mu);
    g_conv_kept.clear();
    g_conv_count.store(0, std::memory_order_release);
}

bool conv_implicit_applies(const ConvGeom &g, bt_code code) {
    if (const char *env = std::getenv("BT_CONV_IMPLICIT")) {
        if (std::strcmp(env, "0") == 0) return false;
    }
    ConvGeom q = g;
    q.O = kBM;                      // the plan's feasibility does not depend on O
    ConvPlan p;
    return plan_conv(q, code, 148, 4, p);   // 4-byte outputs need the most staging
}

cudaError_t launch_tc_conv_implicit(const uint8_t *xp, const uint8_t *wp, bt_code code, const ConvGeom &g, float alpha,
                                    void *out, bt_dtype out_t, unsigned int *err, cudaStream_t s,
                                    const float *scales, bool after_own_pack) {
    if (!conv_implicit_applies(g, code)) return cudaErrorNotSupported;
    ConvPlan p;
    if (!choose_plan(g, code, device_sm_count(), out_t == BT_BF16 || out_t == BT_F16 ? 2 : 4, p))
        return cudaErrorNotSupported;
    p.a.alpha = alpha;
    p.a.scales = scales;
    p.a.out = out;
    p.a.err = err;
    p.a.wait_ns = wait_limit_ns();
    p.a.a_early = after_own_pack ? 1 : 0;
    CUtensorMap ma, mb;
    if (!encode_maps(g, code, p.a, xp, wp, &ma, &mb)) return cudaErrorInvalidValue;
    return launch_code<void>(ma, mb, p, code, out_t, s);
}

bool conv_fused_applies(const ConvGeom &g, bt_code code, bt_dtype x_dtype) {
    // measured on GB300 against the pack kernel + the contraction of packed
    // pixels (ResNet 3x3 layers, stride 1 and 2): the six packing warps of a
    // CTA, beside its MMA and epilogue warps, convert x more slowly than the
    // standalone pack kernel does with the whole GPU, so the two-kernel route
    // is the default and BT_CONV_FUSED=1 turns this one on
    // (or a forced plan that packs x itself, where the environment is silent)
    const char *env = std::getenv("BT_CONV_FUSED");
    if (env != nullptr ? std::strcmp(env, "1") != 0 : !(t_conv_force != nullptr && t_conv_force->fused == 1))
        return false;
    if (x_dtype != BT_F32 && x_dtype != BT_BF16 && x_dtype != BT_F16) return false;
    // every channel plane 16-byte aligned; pixel indices of a plane in 31 bits
    const int64_t hw = g.H * g.W;
    if ((hw * dtype_bytes(x_dtype)) % 16 != 0 || hw >= (int64_t(1) << 30)) return false;
    // element offsets within one image in 32 bits
    if (g.C * hw >= (int64_t(1) << 31)) return false;
    return conv_implicit_applies(g, code);
}

cudaError_t launch_tc_conv_fused(const void *x, bt_dtype x_dtype, const float *bias, int64_t bias_len,
                                 const uint8_t *wp, bt_code code, const ConvGeom &g, float alpha, void *out,
                                 bt_dtype out_t, unsigned int *err, cudaStream_t s, const float *scales) {
    if (!conv_fused_applies(g, code, x_dtype)) return cudaErrorNotSupported;
    ConvPlan p;
    if (!choose_plan(g, code, device_sm_count(), out_t == BT_BF16 || out_t == BT_F16 ? 2 : 4, p))
        return cudaErrorNotSupported;
    plan_fused(g, code, p);
    p.a.alpha = alpha;
    p.a.scales = scales;
    p.a.out = out;
    p.a.err = err;
    p.a.wait_ns = wait_limit_ns();
    p.a.x = x;
    p.a.bias = bias;
    p.a.bias_len = static_cast<int>(bias_len);
    // the weights' map only: the pixel-map slot is not read (the weights' map fills it)
    CUtensorMap ma;
    if (!encode_weight_map(g, code, p.a, wp, &ma)) return cudaErrorInvalidValue;
    switch (x_dtype) {
        case BT_F32: return launch_fused_f32(ma, p, code, out_t, s);
        case BT_F16: return launch_fused_f16(ma, p, code, out_t, s);
        default: return launch_fused_bf16(ma, p, code, out_t, s);
    }
}

}  // namespace bt
