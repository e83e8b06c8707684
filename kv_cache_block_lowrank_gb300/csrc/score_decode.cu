// score_decode.cu -- host side of the decode scorer: shape checks, launch layout (warps,
// shared memory, bulk-copy slots, the fused ranking's mode) and dispatch to the per-r kernel
// instances of score_decode_k{1,2,4,8}.cu.  The kernel itself is in score_decode_kernel.cuh.
#include "score_decode_kernel.cuh"

HSS_DECODE_INSTANCES(extern, 1)
HSS_DECODE_INSTANCES(extern, 2)
HSS_DECODE_INSTANCES(extern, 4)
HSS_DECODE_INSTANCES(extern, 8)

namespace hss {
using namespace decode;
namespace {

int frag_bytes_per_warp(const ScoreArgs& a) {
    const int ksteps = a.r / 16;
    const int nvec = a.rows_per_seq * (a.num_q_heads / a.num_kv_heads);
    const int nt = (nvec + 7) / 8;
    return a.num_kv_heads * ksteps * nt * 32 * 8;
}

// Shared memory of the in-kernel query projection: every sequence's fragment cache, P's
// fragments, then the query rows.
int64_t inline_bytes(const ScoreArgs& a, int32_t head_dim) {
    const int64_t q_rows = static_cast<int64_t>(a.num_seqs) * a.rows_per_seq * a.num_q_heads;
    return static_cast<int64_t>(a.num_seqs) * frag_bytes_per_warp(a) +
           static_cast<int64_t>(a.r) * head_dim * 2 + q_rows * (head_dim + 32) * 2;
}

}  // namespace

bool score_decode_supported(const ScoreArgs& a) {
    if (a.block_size % 16 != 0 || a.r % 16 != 0) return false;
    const int ksteps = a.r / 16;
    if (ksteps != 1 && ksteps != 2 && ksteps != 4 && ksteps != 8) return false;
    const int64_t nvec = static_cast<int64_t>(a.rows_per_seq) * (a.num_q_heads / a.num_kv_heads);
    if (nvec < 1 || nvec > 16) return false;
    return frag_bytes_per_warp(a) <= kFragBudgetBytes;
}

bool score_decode_inline_supported(const ScoreArgs& a, int32_t head_dim) {
    if (!score_decode_supported(a) || a.num_seqs < 1 || a.num_seqs > kInlineMaxSeqs) return false;
    if (head_dim % 32 != 0 || a.ctx_len != nullptr || a.row_pos0 != nullptr) return false;
    return inline_bytes(a, head_dim) <= kInlineBudgetBytes;
}

hss_status launch_score_decode(const ScoreArgs& a, cudaStream_t stream, const FusedRank* fr,
                               bool* fused, const InlineQ* iq) {
    if (fused != nullptr) *fused = false;
    if (a.total == 0) return HSS_OK;
    const DeviceInfo* dev = current_device_info();
    if (dev == nullptr) return HSS_ERR_CUDA;
    if (!score_decode_supported(a)) return HSS_ERR_UNSUPPORTED_SHAPE;
    DecodeParams p;
    p.Qp = a.Qp;
    p.A_g = a.A_g;
    p.table = a.table;
    p.seq_offsets = a.seq_offsets;
    p.scores = a.scores;
    p.dev_status = a.dev_status;
    p.lib_error = dev->error_word;
    p.layer_slots = a.layer_offset_slots;
    p.max_blocks = a.max_blocks;
    p.total = a.total;
    p.num_seqs = a.num_seqs;
    p.rows = a.rows_per_seq;
    p.nq = a.num_q_heads;
    p.nkv = a.num_kv_heads;
    p.r = a.r;
    p.bs = a.block_size;
    p.g = a.num_q_heads / a.num_kv_heads;
    p.nvec = a.rows_per_seq * p.g;
    p.counters = nullptr;
    p.victims = nullptr;
    p.k = 0;
    p.sel_cap = 0;
    p.todo_cap = 0;
    p.new_ids = nullptr;
    p.num_new = 0;
    p.early = 0;
    p.ctx_len = a.ctx_len;
    p.row_pos0 = a.row_pos0;
    p.Q = nullptr;
    p.P = nullptr;
    p.hd = 0;
    p.cache_bytes = 0;
    p.nowait = 0;
    p.tma_bar_off = 0;
    p.tma_buf_off = 0;
    p.wait_limit_ns = fr != nullptr && fr->wait_limit_ns > 0
                          ? static_cast<uint64_t>(fr->wait_limit_ns) : kWaitLimitNs;
    p.withhold_cta = fr != nullptr ? fr->withhold_cta : -1;
    if (fr != nullptr && fr->early && fr->num_new <= 64) {
        p.new_ids = fr->new_ids;
        p.num_new = static_cast<int32_t>(fr->num_new);
        p.early = 1;
    }

    const int fb = frag_bytes_per_warp(a);
    int warps_per_cta = std::max(1, std::min(kWarpsMax, kFragBudgetBytes / fb));
    int smem = warps_per_cta * fb;
    if (iq != nullptr) {
        if (!score_decode_inline_supported(a, iq->head_dim)) return HSS_ERR_UNSUPPORTED_SHAPE;
        p.Q = iq->Q;
        p.P = iq->P;
        p.hd = iq->head_dim;
        p.cache_bytes = a.num_seqs * fb;
        p.nowait = iq->nowait && p.early && p.num_new <= 32 ? 1 : 0;
        warps_per_cta = kWarpsMax;
        smem = static_cast<int>(inline_bytes(a, iq->head_dim));
    }
    // Enough warps for two CTAs per SM; each warp takes a contiguous run of entries.
    const int64_t target_warps = static_cast<int64_t>(dev->num_sms) * 2 * warps_per_cta;
    p.entries_per_warp = std::max<int64_t>(1, (a.total + target_warps - 1) / target_warps);
    // Queries projected in the scorer, at most two entries per warp and small slots: the
    // slots come by bulk copies into one shared buffer per warp (eight mbarriers, then the
    // buffers on 128-byte boundaries), if that still leaves room for two CTAs per SM.
    const int64_t slot_bytes = static_cast<int64_t>(a.num_kv_heads) * a.block_size * a.r * 2;
    if (iq != nullptr && p.entries_per_warp <= kTmaMaxEntriesPerWarp &&
        slot_bytes <= kTmaMaxSlotBytes) {
        const int bar_off = (smem + 15) / 16 * 16;
        const int buf_off = (bar_off + 8 * kWarpsMax + 127) / 128 * 128;
        const int end = buf_off + kWarpsMax * static_cast<int>(slot_bytes);
        if (end + 8 * 1024 <= dev->max_smem_optin / 2) {
            p.tma_bar_off = bar_off;
            p.tma_buf_off = buf_off;
            smem = end;
        }
    }
    p.frag_bytes_cta = smem;
    const int64_t warps = (a.total + p.entries_per_warp - 1) / p.entries_per_warp;
    const int grid = static_cast<int>((warps + warps_per_cta - 1) / warps_per_cta);
    // The ranking can ride along when a whole CTA of 8 warps is there to run it, every
    // sequence's keys fit in shared memory and the extra shared memory stays modest.
    // Long sequences are ranked by the dedicated kernel (1024 threads) instead.
    const int ksteps = a.r / 16;
    const int nt = (p.nvec + 7) / 8;
    p.spread = 0;
    if (fr != nullptr && fr->spread_region != nullptr && warps_per_cta == kWarpsMax &&
        a.num_seqs >= 1 && a.num_seqs <= kSpreadMaxSeqs && a.total <= kSpreadMaxEntries &&
        (reinterpret_cast<uintptr_t>(fr->spread_region) & 15u) == 0 && p.frag_bytes_cta % 16 == 0 &&
        p.entries_per_warp * warps_per_cta <= kSpreadMaxCta) {
        // Spread ranking needs the whole grid resident at once (its CTAs wait for each other).
        const int todo_cap = static_cast<int>(p.entries_per_warp * warps_per_cta);
        // ... then the call tag, the sequence offsets and the entries' sequence indices.
        const int smem_spread = smem + 4 * todo_cap + 4 * kWarpsMax * kSpreadMaxCta + 16 +
                                4 * (kSpreadMaxSeqs + 1) + kSpreadMaxCta + 12;
        int per_sm = 0;
#define HSS_DECODE_CASE(KS, NT_) \
    if (ksteps == KS && nt == NT_) per_sm = ctas_per_sm_t<KS, NT_>(p, smem_spread);
        HSS_DECODE_CASE(1, 1)
        HSS_DECODE_CASE(1, 2)
        HSS_DECODE_CASE(2, 1)
        HSS_DECODE_CASE(2, 2)
        HSS_DECODE_CASE(4, 1)
        HSS_DECODE_CASE(4, 2)
        HSS_DECODE_CASE(8, 1)
        HSS_DECODE_CASE(8, 2)
#undef HSS_DECODE_CASE
        if (static_cast<int64_t>(per_sm) * dev->num_sms >= grid) {
            p.spread = 1;
            p.todo_cap = todo_cap;
            p.counters = fr->spread_region;  // the tail's call number and tagged words
            p.victims = fr->victims;
            p.k = fr->k;
            smem = smem_spread;
            if (fused != nullptr) *fused = true;
        }
    }
    if (fr != nullptr && fr->require_spread && !p.spread) return HSS_ERR_UNSUPPORTED_SHAPE;
    if (!p.spread && fr != nullptr && fr->counters != nullptr && warps_per_cta == kWarpsMax &&
        a.total <= kWarpsMax * 32 * rankdev::keys_per_thread<kWarpsMax * 32>()) {
        const int sel_cap = rankdev::rank_sel_cap(fr->k);
        const int todo_cap = static_cast<int>(p.entries_per_warp * warps_per_cta);
        const int extra = rankdev::rank_smem_bytes(sel_cap) + (todo_cap + 1) * 4;
        if (smem + extra <= 100 * 1024) {
            p.todo_cap = todo_cap;
            p.counters = fr->counters;
            p.victims = fr->victims;
            p.k = fr->k;
            p.sel_cap = sel_cap;
            smem += extra;
            if (fused != nullptr) *fused = true;
        }
    }

#define HSS_DECODE_CASE(KS, NT_)                                                        \
    if (ksteps == KS && nt == NT_) return launch_t<KS, NT_>(p, warps_per_cta, smem, grid, stream);
    HSS_DECODE_CASE(1, 1)
    HSS_DECODE_CASE(1, 2)
    HSS_DECODE_CASE(2, 1)
    HSS_DECODE_CASE(2, 2)
    HSS_DECODE_CASE(4, 1)
    HSS_DECODE_CASE(4, 2)
    HSS_DECODE_CASE(8, 1)
    HSS_DECODE_CASE(8, 2)
#undef HSS_DECODE_CASE
    return HSS_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace hss
