// api.cu -- the C ABI (include/resolvent.h): argument checks, workspace layout, per-head
// dispatch and launches on the caller's stream. No allocation, no synchronisation (except
// resolvent_status_sync).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "resolvent.h"
#include "resolvent_internal.h"

using namespace rs;

namespace {

thread_local int g_launches = 0;
uint64_t g_wait_limit_ns = kWaitLimitNs;
int g_chain_withhold = -1;
int g_position_withhold = -1;
int g_head_withhold = -1;
int g_operator_withhold_stats = -1, g_operator_withhold_write = -1;

// Optional timing of the main kernels of each call: CUDA event pairs recorded on the caller's
// stream around each class of launch (RS_PROF_* in resolvent.h), kept in order.
constexpr int kProfSlots = 4096;
struct Prof {
    bool on = false;
    int next = 0;
    cudaEvent_t ev[kProfSlots][2];
    int kind[kProfSlots];
    bool made = false;
} g_prof;
std::mutex g_prof_mu;

void prof_mark(cudaStream_t s, int which, int kind)
{
    if (!g_prof.on || g_prof.next >= kProfSlots) return;
    cudaEventRecord(g_prof.ev[g_prof.next][which], s);
    g_prof.kind[g_prof.next] = kind;
    if (which == 1) ++g_prof.next;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int pad64(int x) { return x <= 64 ? 64 : 128; }


rs_status check_switches(const rs_switches &sw, int H)
{
    if (!sw.beta || !sw.qk || !sw.g) return RS_ERR_SHAPE;
    if (!(sw.count == 1 || sw.count == H)) return RS_ERR_SHAPE;
    for (int i = 0; i < sw.count; ++i)
        if (!std::isfinite(sw.beta[i]) || !std::isfinite(sw.qk[i]) || !std::isfinite(sw.g[i]))
            return RS_ERR_NONFINITE;  // a non-finite switch is refused
    return RS_OK;
}

struct Sw {
    float beta, qk, g;
};
Sw sw_of(const rs_switches &sw, int h)
{
    const int i = sw.count == 1 ? 0 : h;
    return {sw.beta[i], sw.qk[i], sw.g[i]};
}

// Heads (b, h) selected by `pred`, in chunks of at most kMaxSlots per table.
template <typename Pred>
std::vector<HeadTable> tables_for(const rs_switches &sw, int B, int H, Pred pred)
{
    std::vector<HeadTable> out;
    HeadTable t;
    std::memset(&t, 0, sizeof(t));
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const Sw s = sw_of(sw, h);
            if (!pred(s)) continue;
            t.bh[t.count] = b * H + h;
            t.beta[t.count] = s.beta;
            t.qk[t.count] = s.qk;
            t.g[t.count] = s.g;
            if (++t.count == kMaxSlots) {
                out.push_back(t);
                std::memset(&t, 0, sizeof(t));
            }
        }
    if (t.count) out.push_back(t);
    return out;
}

// qk = 0: W_ij = G_ij / Z_i^beta with Z_i = sum_{j<=i} R_ij = m_i Z_{i-1} + 1, so
// O_i = y_i Z_i^{-beta} with y the chain over V: an O(n) evaluation for any beta.
bool is_chain_head(const Sw &s) { return s.qk == 0.f; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D view [heads, rows, cols] of a bf16 tensor; boxes of 64 columns x 128 rows x 1 head,
// 128-byte swizzle, rows past `rows` read as zeros.
}  // namespace

int rs::device_sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

namespace {

// [heads, rows, cols] row-major, 128-byte swizzled boxes of box_rows rows x 128 bytes:
// bf16 inputs (box 64 x 128) or fp32 outputs (box 32 x box_rows).
bool make_tmap(CUtensorMap *m, const void *base, int cols, int rows, int heads, bool f32 = false,
               unsigned box_rows = 128)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)cols * es, (cuuint64_t)rows * cols * es};
    cuuint32_t box[3] = {f32 ? 32u : 64u, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Workspace of resolvent_head_forward.
struct HeadWs {
    size_t gate, prefix, suffix, carry, numkv, qpad, kpad, vpad, chain, total;
    bool copy_qk, copy_v;
};

HeadWs head_ws(int B, int H, int n, int d, int dv, rs_dtype dt)
{
    HeadWs w{};
    const size_t BH = (size_t)B * H, tok = BH * n, nb = (size_t)(n + kBlock - 1) / kBlock;
    w.copy_qk = dt == RS_F32 || d != pad64(d);
    w.copy_v = dt == RS_F32 || dv != pad64(dv);
    size_t off = 0;
    w.gate = off; off += up256(tok * 8);
    w.prefix = off; off += up256(tok * 8);
    w.suffix = off; off += up256(tok * 8);
    w.carry = off; off += up256(BH * nb * 8);
    w.numkv = off; off += up256(std::min<size_t>(BH, kMaxSlots) * nb * 4);
    w.qpad = off; off += w.copy_qk ? up256(tok * pad64(d) * 2) : 0;
    w.kpad = off; off += w.copy_qk ? up256(tok * pad64(d) * 2) : 0;
    w.vpad = off; off += w.copy_v ? up256(tok * pad64(dv) * 2) : 0;
    w.chain = off; off += up256(chain_scratch_bytes((int)std::min<size_t>(BH, kMaxSlots), n, dv));
    w.total = off;
    return w;
}

struct ChainWs {
    int *counter, *flags;
    float2 *agg_a, *agg_y, *incl_y, *agg_z;
    float *incl_z;
    size_t zero_bytes;
};

ChainWs chain_ws(void *base, int slots, int n, int dv)
{
    const size_t nchunks = (size_t)(n + kChainChunk - 1) / kChainChunk;
    const size_t chunks = (size_t)slots * nchunks;
    char *p = static_cast<char *>(base);
    ChainWs w;
    w.counter = reinterpret_cast<int *>(p);
    w.flags = w.counter + 1;
    w.zero_bytes = sizeof(int) * (chunks + 1);
    p += up256(sizeof(int) * (chunks + 1));
    w.agg_a = reinterpret_cast<float2 *>(p);
    p += up256(sizeof(float2) * chunks);
    w.agg_y = reinterpret_cast<float2 *>(p);
    p += up256(sizeof(float2) * chunks * dv);
    w.incl_y = reinterpret_cast<float2 *>(p);
    p += up256(sizeof(float2) * chunks * dv);
    w.agg_z = reinterpret_cast<float2 *>(p);
    p += up256(sizeof(float2) * chunks);
    w.incl_z = reinterpret_cast<float *>(p);
    return w;
}

rs_status run_chain(const std::vector<HeadTable> &tabs, const float *u, const float *theta,
                    const void *b, int b_is_bf16, int n, int dv, float *y_re, float *y_im,
                    void *scratch, int32_t *status, cudaStream_t s, int prof_kind, bool normalize = false,
                    const float2 *carry_in = nullptr, float2 *carry_out = nullptr)
{
    for (size_t i = 0; i < tabs.size(); ++i) {
        const HeadTable &t = tabs[i];
        ChainWs w = chain_ws(scratch, t.count, n, dv);
        cudaError_t e = cudaMemsetAsync(w.counter, 0, w.zero_bytes, s);
        if (e != cudaSuccess) return RS_ERR_CUDA;
        ChainArgs a{};
        a.u = u; a.theta = theta; a.b = b; a.b_is_bf16 = b_is_bf16; a.n = n; a.dv = dv;
        a.y_re = y_re; a.y_im = y_im; a.counter = w.counter; a.flags = w.flags;
        a.agg_a = w.agg_a; a.agg_y = w.agg_y; a.incl_y = w.incl_y; a.status = status;
        a.normalize = normalize ? 1 : 0; a.agg_z = w.agg_z; a.incl_z = w.incl_z;
        a.carry_in = carry_in; a.carry_out = carry_out;
        a.wait_limit_ns = g_wait_limit_ns; a.withhold_chunk = g_chain_withhold;
        if (i == 0) prof_mark(s, 0, prof_kind);
        e = launch_chain_scan(a, t, s);
        if (i + 1 == tabs.size()) prof_mark(s, 1, prof_kind);
        ++g_launches;
        if (e != cudaSuccess) return RS_ERR_CUDA;
    }
    return RS_OK;
}

}  // namespace

extern "C" {

const char *resolvent_status_string(rs_status s)
{
    switch (s) {
    case RS_OK: return "ok";
    case RS_ERR_NONFINITE: return "non-finite input refused";
    case RS_ERR_SHAPE: return "shape error";
    case RS_ERR_UNSUPPORTED: return "unsupported size";
    case RS_ERR_ALIGN: return "pointer not 16-byte aligned";
    case RS_ERR_WORKSPACE: return "workspace missing or too small";
    case RS_ERR_CUDA: return "CUDA runtime error";
    case RS_ERR_TIMEOUT: return "a bounded device wait ran out";
    }
    return "unknown status";
}

int resolvent_last_launch_count(void) { return g_launches; }

rs_status resolvent_gate_prep(const float *u, const float *theta, rs_switches sw, int B, int H,
                              int n, float *m, float *theta_p, float *gate, float *prefix,
                              float *suffix, float *block_carry, int32_t *status_dev,
                              void *stream)
{
    g_launches = 0;
    if (B < 0 || H < 0 || n < 0) return RS_ERR_SHAPE;
    if ((size_t)B * H == 0 || n == 0) return RS_OK;
    rs_status st = check_switches(sw, H);
    if (st != RS_OK) return st;
    if (!u || !theta || !status_dev) return RS_ERR_SHAPE;
    for (const void *p : {(const void *)u, (const void *)theta, (const void *)m, (const void *)theta_p,
                          (const void *)gate, (const void *)prefix, (const void *)suffix,
                          (const void *)block_carry})
        if (p && !aligned16(p)) return RS_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const auto tabs = tables_for(sw, B, H, [](const Sw &) { return true; });
    prof_mark(s, 0, RS_PROF_GATE_PREP);  // after the host-side tables: the pair brackets the launches
    for (const HeadTable &t : tabs) {
        GatePrepArgs a{};
        a.u = u; a.theta = theta; a.n = n; a.m = m; a.theta_p = theta_p;
        a.gate = reinterpret_cast<float2 *>(gate);
        a.prefix = reinterpret_cast<float2 *>(prefix);
        a.suffix = reinterpret_cast<float2 *>(suffix);
        a.carry = reinterpret_cast<float2 *>(block_carry);
        a.status = status_dev; a.write_ungated = 1;
        if (launch_gate_prep(a, t, s) != cudaSuccess) return RS_ERR_CUDA;
        ++g_launches;
    }
    prof_mark(s, 1, RS_PROF_GATE_PREP);
    return RS_OK;
}

size_t resolvent_head_workspace_bytes(int B, int H, int n, int d, int dv, rs_dtype dtype)
{
    if (B <= 0 || H <= 0 || n <= 0 || d <= 0 || dv <= 0) return 0;
    return head_ws(B, H, n, d, dv, dtype).total;
}

rs_status resolvent_head_forward(const void *q, const void *k, const float *u, const float *theta,
                                 const void *v, rs_switches sw, int B, int H, int n, int d, int dv,
                                 rs_dtype dtype, float *O_re, float *O_im, void *workspace,
                                 size_t workspace_bytes, int32_t *status_dev, void *stream)
{
    g_launches = 0;
    if (B < 0 || H < 0 || n < 0) return RS_ERR_SHAPE;
    if ((size_t)B * H == 0 || n == 0) return RS_OK;  // empty sequence: empty readout
    if (d <= 0 || dv <= 0) return RS_ERR_SHAPE;      // head_dim = 0 with n > 0
    if (d > 128 || dv > 128 || d % 8 != 0) return RS_ERR_UNSUPPORTED;
    if (dtype != RS_F32 && dtype != RS_BF16) return RS_ERR_UNSUPPORTED;
    rs_status st = check_switches(sw, H);
    if (st != RS_OK) return st;
    if (!q || !k || !u || !theta || !v || !O_re || !O_im || !status_dev) return RS_ERR_SHAPE;
    for (const void *p : {q, k, (const void *)u, (const void *)theta, v, (const void *)O_re,
                          (const void *)O_im, (const void *)workspace})
        if (!aligned16(p)) return RS_ERR_ALIGN;
    const HeadWs w = head_ws(B, H, n, d, dv, dtype);
    if (!workspace || workspace_bytes < w.total) return RS_ERR_WORKSPACE;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const int BH = B * H;
    const int DP = pad64(d), DVP = pad64(dv);
    const bool f32 = dtype == RS_F32;

    // gated heads first (their tiles are heavier), then heads with g = 0 (G = 1)
    auto head_tabs = tables_for(sw, B, H, [](const Sw &s) { return !is_chain_head(s) && s.g != 0.f; });
    const auto plain_tabs = tables_for(sw, B, H, [](const Sw &s) { return !is_chain_head(s) && s.g == 0.f; });
    head_tabs.insert(head_tabs.end(), plain_tabs.begin(), plain_tabs.end());
    const auto chain_tabs = tables_for(sw, B, H, [](const Sw &s) { return is_chain_head(s); });
    const auto qk0_tabs = tables_for(sw, B, H, [](const Sw &s) { return s.qk == 0.f; });

    // The refusal covers q and k even where qk = 0 removes them from the logits.
    for (const HeadTable &t : qk0_tabs) {
        cudaError_t e1, e2;
        if (f32) {
            e1 = launch_check_finite_f32(static_cast<const float *>(q), (int64_t)n * d, t, status_dev, s);
            e2 = launch_check_finite_f32(static_cast<const float *>(k), (int64_t)n * d, t, status_dev, s);
        } else {
            e1 = launch_check_finite_bf16(static_cast<const __nv_bfloat16 *>(q), (int64_t)n * d, t, status_dev, s);
            e2 = launch_check_finite_bf16(static_cast<const __nv_bfloat16 *>(k), (int64_t)n * d, t, status_dev, s);
        }
        g_launches += 2;
        if (e1 != cudaSuccess || e2 != cudaSuccess) return RS_ERR_CUDA;
    }

    if (!head_tabs.empty()) {
        float2 *gate = reinterpret_cast<float2 *>(ws + w.gate);
        float2 *prefix = reinterpret_cast<float2 *>(ws + w.prefix);
        float2 *suffix = reinterpret_cast<float2 *>(ws + w.suffix);
        float2 *carry = reinterpret_cast<float2 *>(ws + w.carry);
        const void *qs = q, *ks = k, *vs = v;
        if (w.copy_qk) {
            __nv_bfloat16 *qp = reinterpret_cast<__nv_bfloat16 *>(ws + w.qpad);
            __nv_bfloat16 *kp = reinterpret_cast<__nv_bfloat16 *>(ws + w.kpad);
            if (launch_pad_to_bf16(q, f32, (int64_t)BH * n, d, qp, DP, status_dev, f32, s) != cudaSuccess ||
                launch_pad_to_bf16(k, f32, (int64_t)BH * n, d, kp, DP, status_dev, f32, s) != cudaSuccess)
                return RS_ERR_CUDA;
            g_launches += 2;
            qs = qp;
            ks = kp;
        }
        if (w.copy_v) {
            __nv_bfloat16 *vp = reinterpret_cast<__nv_bfloat16 *>(ws + w.vpad);
            if (launch_pad_to_bf16(v, f32, (int64_t)BH * n, dv, vp, DVP, status_dev, 0, s) != cudaSuccess)
                return RS_ERR_CUDA;
            g_launches += 1;
            vs = vp;
        }
        HeadMaps maps;
        std::memset(&maps, 0, sizeof(maps));
        if (!make_tmap(&maps.q, qs, DP, n, BH) || !make_tmap(&maps.k, ks, DP, n, BH) ||
            !make_tmap(&maps.v, vs, DVP, n, BH))
            return RS_ERR_CUDA;
        // the outputs leave by 16-byte stores when their rows are a multiple of 16 bytes
        const bool tma_out = dv % 4 == 0;
        std::vector<HeadArgs> args;
        for (const HeadTable &t : head_tabs) {
            HeadArgs ha{};
            ha.n = n; ha.d = d; ha.dv = dv; ha.gate = gate; ha.prefix = prefix; ha.suffix = suffix;
            ha.carry = carry; ha.O_re = O_re; ha.O_im = O_im; ha.status = status_dev;
            ha.tma_out = tma_out ? 1 : 0;
            ha.numkv = reinterpret_cast<int *>(ws + w.numkv);
            ha.withhold = g_head_withhold;
            // one block per SM: the block that starts about when this one ends is one SM count on
            ha.prefetch_ahead = device_sm_count();
            // about 24 MB of K and V per head group: a group's K/V tiles stay in L2
            const size_t kv_head = (size_t)n * (DP + DVP) * 2;
            ha.heads_per_group = (int)std::max<size_t>(1, std::min<size_t>(t.count, (24u << 20) / kv_head));
            args.push_back(ha);
        }
        for (const HeadTable &t : head_tabs) {
            GatePrepArgs ga{};
            ga.u = u; ga.theta = theta; ga.n = n; ga.gate = gate; ga.prefix = prefix;
            ga.suffix = suffix; ga.carry = carry; ga.status = status_dev; ga.write_ungated = 0;
            if (launch_gate_prep(ga, t, s) != cudaSuccess) return RS_ERR_CUDA;
            ++g_launches;
        }
        // The per-tile key-tile counts share one scratch array, so each table's count runs
        // right before its head launch (same stream).
        for (size_t i = 0; i < head_tabs.size(); ++i) {
            const int kind = head_tabs[i].g[0] != 0.f ? RS_PROF_HEAD_GATED : RS_PROF_HEAD_REAL;
            prof_mark(s, 0, kind);
            if (head_tabs[i].g[0] != 0.f) {
                if (launch_head_numkv(args[i], head_tabs[i], s) != cudaSuccess) return RS_ERR_CUDA;
                ++g_launches;
            }
            if (launch_head_fwd(args[i], head_tabs[i], maps, DP, DVP, s) != cudaSuccess) return RS_ERR_CUDA;
            prof_mark(s, 1, kind);
            ++g_launches;
        }
    }

    // qk = 0 and beta = 0: W = G exactly, so O is the chain over V.
    if (!chain_tabs.empty()) {
        st = run_chain(chain_tabs, u, theta, v, f32 ? 0 : 1, n, dv, O_re, O_im, ws + w.chain,
                       status_dev, s, RS_PROF_READOUT, true);
        if (st != RS_OK) return st;
    }
    return RS_OK;
}

// Workspace of resolvent_operator.
struct OperatorWs {
    size_t gate, prefix, suffix, carry, qpad, kpad, part, ctab, rowf, rowq, total;
    bool copy_qk;
};

OperatorWs operator_ws(int B, int H, int n, int d, rs_dtype dt)
{
    OperatorWs w{};
    const size_t BH = (size_t)B * H, tok = BH * n, nb = (size_t)(n + kBlock - 1) / kBlock;
    const size_t slots = std::min<size_t>(BH, kMaxSlots);
    const size_t nch = (nb + operator_chunk(n) - 1) / operator_chunk(n);
    w.copy_qk = dt == RS_F32 || d != pad64(d);
    size_t off = 0;
    w.gate = off; off += up256(tok * 8);
    w.prefix = off; off += up256(tok * 8);
    w.suffix = off; off += up256(tok * 8);
    w.carry = off; off += up256(BH * nb * 8);
    w.qpad = off; off += w.copy_qk ? up256(tok * pad64(d) * 2) : 0;
    w.kpad = off; off += w.copy_qk ? up256(tok * pad64(d) * 2) : 0;
    w.part = off; off += up256(slots * nb * nch * 128 * 8);
    w.ctab = off; off += up256(slots * nb * nb * 8);
    w.rowf = off; off += up256(slots * nb * 128 * 16);
    w.rowq = off; off += up256(slots * nb * 128 * 4);
    w.total = off;
    return w;
}

size_t resolvent_operator_workspace_bytes(int B, int H, int n, int d, rs_dtype dtype)
{
    if (B <= 0 || H <= 0 || n <= 0 || d <= 0) return 0;
    return operator_ws(B, H, n, d, dtype).total;
}

rs_status resolvent_operator(const void *q, const void *k, const float *u, const float *theta,
                             rs_switches sw, int B, int H, int n, int d, rs_dtype dtype,
                             float *W_re, float *W_im, void *workspace, size_t workspace_bytes,
                             int32_t *status_dev, void *stream)
{
    g_launches = 0;
    if (B < 0 || H < 0 || n < 0) return RS_ERR_SHAPE;
    if ((size_t)B * H == 0 || n == 0) return RS_OK;
    if (d <= 0) return RS_ERR_SHAPE;
    if (d > 128 || d % 8 != 0) return RS_ERR_UNSUPPORTED;
    if (dtype != RS_F32 && dtype != RS_BF16) return RS_ERR_UNSUPPORTED;
    rs_status st = check_switches(sw, H);
    if (st != RS_OK) return st;
    if (!q || !k || !u || !theta || !W_re || !W_im || !status_dev) return RS_ERR_SHAPE;
    for (const void *p : {q, k, (const void *)u, (const void *)theta, (const void *)W_re,
                          (const void *)W_im, (const void *)workspace})
        if (!aligned16(p)) return RS_ERR_ALIGN;
    const OperatorWs w = operator_ws(B, H, n, d, dtype);
    if (!workspace || workspace_bytes < w.total) return RS_ERR_WORKSPACE;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const int BH = B * H, DP = pad64(d);
    const bool f32 = dtype == RS_F32;
    auto tabs = tables_for(sw, B, H, [](const Sw &s) { return s.g != 0.f; });
    const auto plain = tables_for(sw, B, H, [](const Sw &s) { return s.g == 0.f; });
    tabs.insert(tabs.end(), plain.begin(), plain.end());
    float2 *gate = reinterpret_cast<float2 *>(ws + w.gate);
    float2 *prefix = reinterpret_cast<float2 *>(ws + w.prefix);
    float2 *suffix = reinterpret_cast<float2 *>(ws + w.suffix);
    float2 *carry = reinterpret_cast<float2 *>(ws + w.carry);
    const void *qs = q, *ks = k;
    if (w.copy_qk) {
        __nv_bfloat16 *qp = reinterpret_cast<__nv_bfloat16 *>(ws + w.qpad);
        __nv_bfloat16 *kp = reinterpret_cast<__nv_bfloat16 *>(ws + w.kpad);
        if (launch_pad_to_bf16(q, f32, (int64_t)BH * n, d, qp, DP, status_dev, f32, s) != cudaSuccess ||
            launch_pad_to_bf16(k, f32, (int64_t)BH * n, d, kp, DP, status_dev, f32, s) != cudaSuccess)
            return RS_ERR_CUDA;
        g_launches += 2;
        qs = qp;
        ks = kp;
    }
    OpMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!make_tmap(&maps.q, qs, DP, n, BH) || !make_tmap(&maps.k, ks, DP, n, BH)) return RS_ERR_CUDA;
    // W goes out by tensor-map stores when its rows are a multiple of 16 bytes
    const bool tma_out = n % 4 == 0;
    if (tma_out && (!make_tmap(&maps.wre, W_re, n, n, BH, true, 32) ||
                    !make_tmap(&maps.wim, W_im, n, n, BH, true, 32)))
        return RS_ERR_CUDA;
    for (const HeadTable &t : tabs) {
        if (t.g[0] == 0.f) continue;  // G = 1: no gate products
        GatePrepArgs ga{};
        ga.u = u; ga.theta = theta; ga.n = n; ga.gate = gate; ga.prefix = prefix;
        ga.suffix = suffix; ga.carry = carry; ga.status = status_dev; ga.write_ungated = 0;
        if (launch_gate_prep(ga, t, s) != cudaSuccess) return RS_ERR_CUDA;
        ++g_launches;
    }
    for (const HeadTable &t : tabs) {
        OpArgs oa{};
        oa.n = n; oa.d = d; oa.chunk = operator_chunk(n);
        oa.gate = gate; oa.prefix = prefix; oa.suffix = suffix; oa.carry = carry;
        oa.W_re = W_re; oa.W_im = W_im;
        oa.part = reinterpret_cast<float2 *>(ws + w.part);
        oa.ctab = reinterpret_cast<float2 *>(ws + w.ctab);
        oa.rowf = reinterpret_cast<float4 *>(ws + w.rowf);
        oa.rowq = reinterpret_cast<float *>(ws + w.rowq);
        oa.status = status_dev; oa.tma_out = tma_out ? 1 : 0;
        oa.withhold_stats = g_operator_withhold_stats;
        oa.withhold_write = g_operator_withhold_write;
        if (launch_operator_stats(oa, t, maps, DP, s) != cudaSuccess) return RS_ERR_CUDA;
        prof_mark(s, 0, RS_PROF_OPERATOR);
        if (launch_operator(oa, t, maps, DP, s) != cudaSuccess) return RS_ERR_CUDA;
        prof_mark(s, 1, RS_PROF_OPERATOR);
        g_launches += 3;
    }
    return RS_OK;
}

// Row stride of the position kernel table: whole 128-key tiles, plus one more (zeros).
int position_kstride(int n) { return (n + 127) / 128 * 128 + 128; }

// Workspace of resolvent_position_head.
struct PositionWs {
    size_t vpad, kap, C, meta, total;
    bool copy_v;
};

PositionWs position_ws(int B, int H, int n, int dv, rs_dtype dt)
{
    PositionWs w{};
    const size_t BH = (size_t)B * H, tok = BH * n;
    const size_t slots = std::min<size_t>(BH, kMaxSlots);
    w.copy_v = dt == RS_F32 || dv != pad64(dv);
    size_t off = 0;
    w.vpad = off; off += w.copy_v ? up256(tok * pad64(dv) * 2) : 0;
    w.kap = off; off += up256(slots * (size_t)position_kstride(n) * 2);
    w.C = off; off += up256(slots * n * 4);
    w.meta = off; off += up256(slots * 8);
    w.total = off;
    return w;
}

size_t resolvent_position_workspace_bytes(int B, int H, int n, int dv, rs_dtype dtype)
{
    if (B <= 0 || H <= 0 || n <= 0 || dv <= 0) return 0;
    return position_ws(B, H, n, dv, dtype).total;
}

rs_status resolvent_position_head(const float *a, const void *v, rs_switches sw, int B, int H, int n,
                                  int dv, rs_dtype dtype, float *O, void *workspace,
                                  size_t workspace_bytes, int32_t *status_dev, void *stream)
{
    g_launches = 0;
    if (B < 0 || H < 0 || n < 0) return RS_ERR_SHAPE;
    if ((size_t)B * H == 0 || n == 0) return RS_OK;
    if (dv <= 0) return RS_ERR_SHAPE;
    if (dv > 128) return RS_ERR_UNSUPPORTED;
    if (dtype != RS_F32 && dtype != RS_BF16) return RS_ERR_UNSUPPORTED;
    rs_status st = check_switches(sw, H);
    if (st != RS_OK) return st;
    for (int h = 0; h < H; ++h)  // the position-only form has no gates
        if (sw_of(sw, h).g != 0.f) return RS_ERR_UNSUPPORTED;
    if (!a || !v || !O || !status_dev) return RS_ERR_SHAPE;
    for (const void *p : {(const void *)a, v, (const void *)O, (const void *)workspace})
        if (!aligned16(p)) return RS_ERR_ALIGN;
    const PositionWs w = position_ws(B, H, n, dv, dtype);
    if (!workspace || workspace_bytes < w.total) return RS_ERR_WORKSPACE;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const int BH = B * H, DVP = pad64(dv);
    const bool f32 = dtype == RS_F32;
    const void *vs = v;
    if (w.copy_v) {
        __nv_bfloat16 *vp = reinterpret_cast<__nv_bfloat16 *>(ws + w.vpad);
        if (launch_pad_to_bf16(v, f32, (int64_t)BH * n, dv, vp, DVP, status_dev, 0, s) != cudaSuccess)
            return RS_ERR_CUDA;
        g_launches += 1;
        vs = vp;
    }
    PosMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!make_tmap(&maps.v, vs, DVP, n, BH)) return RS_ERR_CUDA;
    for (const HeadTable &t : tables_for(sw, B, H, [](const Sw &) { return true; })) {
        PosArgs pa{};
        pa.n = n; pa.H = H; pa.dv = dv; pa.a = a;
        pa.kap = reinterpret_cast<__nv_bfloat16 *>(ws + w.kap);
        pa.kstride = position_kstride(n);
        pa.C = reinterpret_cast<float *>(ws + w.C);
        pa.meta = reinterpret_cast<float2 *>(ws + w.meta);
        pa.O = O; pa.status = status_dev; pa.vec_out = dv % 4 == 0 ? 1 : 0;
        pa.withhold = g_position_withhold;
        // about 24 MB of V per head group: a group's V tiles stay in L2
        const size_t v_head = (size_t)n * DVP * 2;
        pa.heads_per_group = (int)std::max<size_t>(1, std::min<size_t>(t.count, (24u << 20) / v_head));
        prof_mark(s, 0, RS_PROF_POSITION);
        if (launch_position_head(pa, t, maps, DVP, s) != cudaSuccess) return RS_ERR_CUDA;
        prof_mark(s, 1, RS_PROF_POSITION);
        g_launches += 2;
    }
    return RS_OK;
}

size_t resolvent_chain_workspace_bytes(int B, int H, int n, int dv)
{
    if (B <= 0 || H <= 0 || n <= 0 || dv <= 0) return 0;
    return chain_scratch_bytes((int)std::min<int64_t>((int64_t)B * H, kMaxSlots), n, dv);
}

rs_status resolvent_chain_scan(const float *u, const float *theta, rs_switches sw, const float *b,
                               int B, int H, int n, int dv, float *y_re, float *y_im,
                               void *workspace, size_t workspace_bytes, int32_t *status_dev,
                               void *stream)
{
    g_launches = 0;
    if (B < 0 || H < 0 || n < 0) return RS_ERR_SHAPE;
    if ((size_t)B * H == 0 || n == 0) return RS_OK;
    if (dv <= 0) return RS_ERR_SHAPE;
    if (dv > 128) return RS_ERR_UNSUPPORTED;
    rs_status st = check_switches(sw, H);
    if (st != RS_OK) return st;
    if (!u || !theta || !b || !y_re || !y_im || !status_dev) return RS_ERR_SHAPE;
    for (const void *p : {(const void *)u, (const void *)theta, (const void *)b, (const void *)y_re,
                          (const void *)y_im, (const void *)workspace})
        if (!aligned16(p)) return RS_ERR_ALIGN;
    if (!workspace || workspace_bytes < resolvent_chain_workspace_bytes(B, H, n, dv))
        return RS_ERR_WORKSPACE;
    return run_chain(tables_for(sw, B, H, [](const Sw &) { return true; }), u, theta, b, 0, n, dv,
                     y_re, y_im, workspace, status_dev, static_cast<cudaStream_t>(stream), RS_PROF_CHAIN);
}

rs_status resolvent_chain_scan_carry(const float *u, const float *theta, rs_switches sw,
                                     const float *b, int B, int H, int n, int dv,
                                     const float *carry_in, float *carry_out, float *y_re,
                                     float *y_im, void *workspace, size_t workspace_bytes,
                                     int32_t *status_dev, void *stream)
{
    g_launches = 0;
    if (B < 0 || H < 0 || n < 0) return RS_ERR_SHAPE;
    if ((size_t)B * H == 0 || n == 0) return RS_OK;
    if (dv <= 0) return RS_ERR_SHAPE;
    if (dv > 128) return RS_ERR_UNSUPPORTED;
    rs_status st = check_switches(sw, H);
    if (st != RS_OK) return st;
    if (!u || !theta || !b || !y_re || !y_im || !status_dev) return RS_ERR_SHAPE;
    for (const void *p : {(const void *)u, (const void *)theta, (const void *)b, (const void *)y_re,
                          (const void *)y_im, (const void *)workspace, (const void *)carry_in,
                          (const void *)carry_out})
        if (p && !aligned16(p)) return RS_ERR_ALIGN;
    if (!workspace || workspace_bytes < resolvent_chain_workspace_bytes(B, H, n, dv))
        return RS_ERR_WORKSPACE;
    // the tables hold at most kMaxSlots heads each; carries are indexed by (b, h) directly
    return run_chain(tables_for(sw, B, H, [](const Sw &) { return true; }), u, theta, b, 0, n, dv,
                     y_re, y_im, workspace, status_dev, static_cast<cudaStream_t>(stream), RS_PROF_CHAIN,
                     false, reinterpret_cast<const float2 *>(carry_in),
                     reinterpret_cast<float2 *>(carry_out));
}

rs_status resolvent_chain_scan_noalloc(const float *u, const float *theta, rs_switches sw,
                                       const float *b, int B, int H, int n, int dv, float *y_re,
                                       float *y_im, int32_t *status_dev, void *stream)
{
    g_launches = 0;
    if (B < 0 || H < 0 || n < 0) return RS_ERR_SHAPE;
    if ((size_t)B * H == 0 || n == 0) return RS_OK;
    if (dv <= 0) return RS_ERR_SHAPE;
    if (dv > 128) return RS_ERR_UNSUPPORTED;
    rs_status st = check_switches(sw, H);
    if (st != RS_OK) return st;
    if (!u || !theta || !b || !y_re || !y_im || !status_dev) return RS_ERR_SHAPE;
    for (const void *p : {(const void *)u, (const void *)theta, (const void *)b, (const void *)y_re,
                          (const void *)y_im})
        if (!aligned16(p)) return RS_ERR_ALIGN;
    if (resolvent_chain_workspace_bytes(B, H, n, dv) > kChainNoAllocBytes)
        return RS_ERR_UNSUPPORTED;  // beyond the fixed scratch
    void *scratch = nullptr;
    if (chain_noalloc_scratch(&scratch) != cudaSuccess) return RS_ERR_CUDA;
    return run_chain(tables_for(sw, B, H, [](const Sw &) { return true; }), u, theta, b, 0, n, dv,
                     y_re, y_im, scratch, status_dev, static_cast<cudaStream_t>(stream), RS_PROF_CHAIN);
}

rs_status resolvent_status_sync(int32_t *status_dev, void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t host = 0;
    if (cudaMemcpyAsync(&host, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RS_ERR_CUDA;
    if (cudaMemsetAsync(status_dev, 0, sizeof(int32_t), s) != cudaSuccess) return RS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
    // after a timeout the outputs, and a refusal raised from them, mean nothing: it comes first
    if (host & RS_STATUS_TIMEOUT) return RS_ERR_TIMEOUT;
    if (host & RS_STATUS_NONFINITE) return RS_ERR_NONFINITE;
    return RS_OK;
}

rs_status resolvent_debug_path_product(const float *u, const float *theta, rs_switches sw, int B,
                                       int H, int n, float *G, void *workspace,
                                       size_t workspace_bytes, int32_t *status_dev, void *stream)
{
    g_launches = 0;
    if (B < 0 || H < 0 || n < 0) return RS_ERR_SHAPE;
    if ((size_t)B * H == 0 || n == 0) return RS_OK;
    if (n > 4096) return RS_ERR_UNSUPPORTED;
    rs_status st = check_switches(sw, H);
    if (st != RS_OK) return st;
    const HeadWs w = head_ws(B, H, n, 8, 1, RS_BF16);
    if (!workspace || workspace_bytes < w.carry + up256((size_t)B * H * ((n + kBlock - 1) / kBlock) * 8))
        return RS_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float2 *gate = reinterpret_cast<float2 *>(ws + w.gate);
    float2 *prefix = reinterpret_cast<float2 *>(ws + w.prefix);
    float2 *suffix = reinterpret_cast<float2 *>(ws + w.suffix);
    float2 *carry = reinterpret_cast<float2 *>(ws + w.carry);
    int first = 0;
    for (const HeadTable &t : tables_for(sw, B, H, [](const Sw &) { return true; })) {
        GatePrepArgs ga{};
        ga.u = u; ga.theta = theta; ga.n = n; ga.gate = gate; ga.prefix = prefix;
        ga.suffix = suffix; ga.carry = carry; ga.status = status_dev; ga.write_ungated = 1;
        if (launch_gate_prep(ga, t, s) != cudaSuccess) return RS_ERR_CUDA;
        if (launch_debug_path_product(gate, prefix, suffix, carry, n, t,
                                      reinterpret_cast<float2 *>(G) + (size_t)first * n * n, s) != cudaSuccess)
            return RS_ERR_CUDA;
        g_launches += 2;
        first += t.count;
    }
    return RS_OK;
}

// Test knobs: the bound on device-side waits, and a chain chunk that withholds its carry
// (so the bounded wait can be seen to run out without a hang).
void resolvent_test_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns ? ns : kWaitLimitNs; }
void resolvent_test_set_chain_withhold(int ticket) { g_chain_withhold = ticket; }
void resolvent_test_set_position_withhold(int block) { g_position_withhold = block; }
void resolvent_test_set_head_withhold(int block) { g_head_withhold = block; }
void resolvent_test_set_operator_withhold(int launch, int block)
{
    g_operator_withhold_stats = launch == 0 ? block : -1;
    g_operator_withhold_write = launch == 1 ? block : -1;
}

rs_status resolvent_profile_enable(int on)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (on && !g_prof.made) {
        for (int i = 0; i < kProfSlots; ++i)
            for (int j = 0; j < 2; ++j)
                if (cudaEventCreate(&g_prof.ev[i][j]) != cudaSuccess) return RS_ERR_CUDA;
        g_prof.made = true;
    }
    g_prof.on = on != 0;
    g_prof.next = 0;
    return RS_OK;
}

int resolvent_profile_collect_kinds(float *ms, int *kind, int max)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    int k = 0;
    for (; k < g_prof.next && k < max; ++k) {
        if (cudaEventSynchronize(g_prof.ev[k][1]) != cudaSuccess) return -1;
        if (cudaEventElapsedTime(&ms[k], g_prof.ev[k][0], g_prof.ev[k][1]) != cudaSuccess) return -1;
        if (kind) kind[k] = g_prof.kind[k];
    }
    g_prof.next = 0;
    return k;
}

int resolvent_profile_collect(float *ms, int max) { return resolvent_profile_collect_kinds(ms, nullptr, max); }

}  // extern "C"
