// attnres_api.cu -- the C ABI: argument validation, launch planning and
// workspace sizing for the AttnRes read operator (include/attnres.h).
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "attnres.h"
#include "attnres_testing.h"
#include "kernels.cuh"

namespace attnres {
namespace {

struct DeviceInfo {
    int sm_count = 0;
    int smem_optin = 0;
    int l2_bytes = 0;
};

// Per-device properties, queried once.
bool device_info(DeviceInfo* out) {
    static DeviceInfo cache[64];
    static bool have[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
    if (dev < 64 && have[dev]) {
        *out = cache[dev];
        return true;
    }
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
        return false;
    if (cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return false;
    if (dev < 64) {
        cache[dev] = d;
        have[dev] = true;
    }
    *out = d;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The cluster backward's switch, ATTNRES_BWD_CLUSTER (read on every call, so
// tests can run every form): unset = the planner's choice, "0" = never (the
// one-CTA streaming backward), "<n>" = clusters of n CTAs with resident rows
// (n = 2, 4 or 8), "s<n>" = clusters of n CTAs streaming the rows, "h<n>" =
// the same with two (smaller) CTAs per SM.
struct ClusterChoice {
    int mode;  // -1 planner, 0 off, 1 resident, 2 streaming, 3 streaming with two CTAs per SM
    int cl;
};
ClusterChoice cluster_choice() {
    const char* v = std::getenv("ATTNRES_BWD_CLUSTER");
    if (!v || !v[0]) return {-1, 0};
    if (v[0] == '0' && v[1] == '\0') return {0, 0};
    const bool strm = v[0] == 's', half = v[0] == 'h';
    const int n = std::atoi(strm || half ? v + 1 : v);
    if (n != 2 && n != 4 && n != 8) return {-1, 0};
    return {half ? 3 : (strm ? 2 : 1), n};
}
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

attnres_status check_shape(const attnres_params* p) {
    if (!p) return ATTNRES_ERR_INVALID_ARG;
    if (p->S < 1 || p->S > ATTNRES_MAX_S) return ATTNRES_ERR_INVALID_ARG;
    if (p->D < 8 || p->D > ATTNRES_MAX_D) return ATTNRES_ERR_INVALID_ARG;
    if (p->D % 8 != 0) return ATTNRES_ERR_ALIGNMENT;
    if (p->R < 1 || p->R > p->D) return ATTNRES_ERR_INVALID_ARG;
    if (p->key_offset < 0 || p->key_offset > p->D - p->R) return ATTNRES_ERR_INVALID_ARG;
    if (p->N < 0) return ATTNRES_ERR_INVALID_ARG;
    if (p->out_norm != 0 && p->out_norm != 1) return ATTNRES_ERR_INVALID_ARG;
    if (!std::isfinite(p->eps) || p->eps < 0.0f) return ATTNRES_ERR_INVALID_ARG;
    if (!std::isfinite(p->scale)) return ATTNRES_ERR_INVALID_ARG;
    if (p->src_ld < p->D) return ATTNRES_ERR_INVALID_ARG;
    if (p->src_ld % 8 != 0) return ATTNRES_ERR_ALIGNMENT;
    if (p->N == 0) return ATTNRES_OK;  // nothing is read: pointers may be NULL
    for (int s = 0; s < p->S; ++s) {
        if (!p->src[s]) return ATTNRES_ERR_INVALID_ARG;
        if (!aligned16(p->src[s])) return ATTNRES_ERR_ALIGNMENT;
    }
    return ATTNRES_OK;
}

// fused: the forward also streams one added row per token (block-partial sum).
// addlast: the backward also streams one added gradient row per token.
attnres_status make_plan(const attnres_params* p, Plan* plan, bool fused = false, bool addlast = false) {
    DeviceInfo dev;
    if (!device_info(&dev)) return ATTNRES_ERR_CUDA;
    Plan pl{};
    const int ncv = p->D / 8;
    // 16-byte vectors per thread so that at most 8 consumer warps cover a row
    pl.vpt = ncv <= 256 ? 1 : (ncv <= 512 ? 2 : 4);
    pl.ncw = (ncv + 32 * pl.vpt - 1) / (32 * pl.vpt);
    if (pl.ncw < 1 || pl.ncw > kMaxConsumerWarps) return ATTNRES_ERR_UNSUPPORTED;
    pl.b_vpt = pl.vpt;
    pl.b_ncw = pl.ncw;
    pl.slot_bytes = static_cast<int>(align_up(static_cast<uint32_t>(p->D) * 2u, 128u));
    pl.s_pad = static_cast<int>(align_up(static_cast<uint32_t>(p->S), 4u));
    const int S = p->S;
    const long long sb = pl.slot_bytes;
    const long long optin = dev.smem_optin;
    auto fits = [&](int chunks, int rows, int dy, bool bwd) {
        return make_layout(chunks, rows, pl.slot_bytes, dy, pl.s_pad, bwd).total <= static_cast<uint32_t>(optin);
    };
    auto max_chunks = [&](int rows, int dy, bool bwd) {
        int c = 0;
        while (c < kMaxChunks && fits(c + 1, rows, dy, bwd)) ++c;
        return c;
    };
    // Forward: CTAs that share an SM split its shared memory.  A chunk holds
    // half a token (or less); a softmax group is all chunks but one, which
    // keeps one chunk loading while the group is read (the other CTA on the
    // SM overlaps the rest).
    {
        const int per_sm = fwd_ctas_per_sm(pl.vpt);
        const long long budget = per_sm > 1 ? (optin / per_sm - 1024) : optin;
        auto ffits = [&](int chunks, int rows) {
            return make_layout(chunks, rows, pl.slot_bytes, fused ? kDeltaSlots : 0, pl.s_pad, false).total <=
                   static_cast<uint32_t>(budget);
        };
        const long long fixed =
            make_layout(0, 1, pl.slot_bytes, fused ? kDeltaSlots : 0, pl.s_pad, false).total + 64;
        long long gmax = (budget - fixed) / (2 * sb);
        if (gmax > kMaxGroup) gmax = kMaxGroup;
        if (gmax < 1) gmax = 1;
        const int groups = static_cast<int>((S + gmax - 1) / gmax);
        pl.f_rows = (S + groups - 1) / groups;
        pl.f_chunks = 0;
        while (pl.f_chunks < kMaxChunks && ffits(pl.f_chunks + 1, pl.f_rows)) ++pl.f_chunks;
        if (pl.f_chunks < 2) return ATTNRES_ERR_UNSUPPORTED;
        int gc = pl.f_chunks - 1;
        while (gc > 1 && gc * pl.f_rows > kMaxGroup) --gc;
        pl.f_group = gc * pl.f_rows;
        long long fg = static_cast<long long>(per_sm) * dev.sm_count;
        if (p->N < fg) fg = p->N;
        pl.fgrid = static_cast<int>(fg < 1 ? 1 : fg);
    }
    // Backward: dy ring, then either a resident token (its rows in two
    // chunks, at most ~60% of the ring so the next token can load meanwhile)
    // or streamed chunks (at least four in the ring).
    {
        // dy slots: two tokens in flight (an added gradient row takes a slot too)
        pl.dy_slots = (sb > 8192 && !addlast) ? 2 : 4;
        const long long fixed = make_layout(0, 1, pl.slot_bytes, pl.dy_slots, pl.s_pad, true).total + 64;
        const long long avail = optin - fixed;
        pl.resident = (static_cast<long long>(S) * sb * 10 <= avail * 6) ? 1 : 0;
        if (pl.resident) {
            // One chunk per token when two tokens fit (measured fastest on the
            // long-sequence workload: fewer barrier operations per token),
            // else halves of a token.
            pl.b_rows = (2LL * S * sb <= avail) ? S : (S >= 2 ? (S + 1) / 2 : 1);
        } else {
            long long g = avail / (4 * sb);
            if (g > 16) g = 16;
            if (g < 1) g = 1;
            pl.b_rows = static_cast<int>(g);
        }
        pl.b_chunks = max_chunks(pl.b_rows, pl.dy_slots, true);
        const int per_token = (S + pl.b_rows - 1) / pl.b_rows;
        if (pl.resident && pl.b_chunks < per_token + 1) pl.resident = 0;
        if (!pl.resident && pl.b_chunks < 2) return ATTNRES_ERR_UNSUPPORTED;
    }
    // Narrow resident rows (D <= 2048): two backward CTAs per SM, each with
    // at most four consumer warps (two vectors a thread) and half the shared
    // memory -- a whole token per chunk, one loading while the other is
    // read.  One CTA's barrier, reduction and coefficient phases then overlap
    // the other's loads and stores (measured: S=10 N=32768 D=2048 R=512 with
    // the norm 0.698 -> 0.468 ms, S=16 N=65536 D=1024 1.09 -> 0.69 ms, S=8
    // N=8192 D=2048 0.119 -> 0.105 ms).  Two CTAs of 160 threads at the
    // kernels' 166 registers use 53K of the SM's 64K registers.
    pl.b_per_sm = 1;
    {
        if (pl.resident && ncv <= 256) {
            const int vpt2 = ncv <= 128 ? 1 : 2;
            const int ncw2 = (ncv + 32 * vpt2 - 1) / (32 * vpt2);
            const uint32_t budget = static_cast<uint32_t>(optin / 2 - 1024);
            int ch = 0;
            while (ch < kMaxChunks && make_layout(ch + 1, S, pl.slot_bytes, pl.dy_slots, pl.s_pad, true).total <= budget)
                ++ch;
            if (ch >= 2) {
                pl.b_vpt = vpt2;
                pl.b_ncw = ncw2;
                pl.b_rows = S;
                pl.b_chunks = ch;
                pl.b_per_sm = 2;
            }
        }
    }
    pl.smem_fwd = make_layout(pl.f_chunks, pl.f_rows, pl.slot_bytes, fused ? kDeltaSlots : 0, pl.s_pad, false).total;
    pl.smem_bwd = make_layout(pl.b_chunks, pl.b_rows, pl.slot_bytes, pl.dy_slots, pl.s_pad, true).total;
    pl.b_slot_bytes = pl.slot_bytes;
    const int thr = p->split_n_threshold > 0 ? p->split_n_threshold : ATTNRES_DEFAULT_SPLIT_N;
    pl.split = p->N >= thr ? 1 : 0;
    long long grid = static_cast<long long>(pl.b_per_sm) * dev.sm_count;
    if (p->N < grid) grid = p->N;
    if (grid < 1) grid = 1;
    pl.grid = static_cast<int>(grid);
    pl.cl = 1;
    pl.slice = p->D;
    pl.nparts = pl.grid;
    // Rows too many for one SM: the backward streams them once per pass, and
    // a row's later reads hit L2 only while the rows read in between -- over
    // the whole grid, (tokens in flight) x (one token's rows) -- fit in it.
    // When one CTA per token overflows half the L2 that way, a cluster of cl
    // CTAs shares each token, each owning a D/cl column slice of every row:
    // cl times fewer tokens in flight.  The smallest cluster that brings the
    // reuse distance within 3/4 of the L2 is taken (measured on the deep
    // shape, S=64, D=8192: one CTA 4.15 ms, clusters of 2 / 4 / 8 3.90 / 5.15 /
    // 11.3 ms -- smaller slices add per-token exchange and barrier time).
    // Resident slices (forced by the switch): the smallest cluster whose
    // slices stay in shared memory.
    const ClusterChoice cc = cluster_choice();
    const long long token_bytes = static_cast<long long>(S) * p->D * 2;
    const bool reuse_overflows = (p->N < pl.grid ? p->N : pl.grid) * token_bytes > dev.l2_bytes / 2;
    if (!pl.resident && !addlast && p->N > 0 && cc.mode != 0 && (cc.mode > 0 || reuse_overflows)) {
        auto try_cluster = [&](int cl, bool resident, int per_sm, Plan* out) -> bool {
            if (p->D % (8 * cl) != 0) return false;
            Plan c = pl;
            c.cl = cl;
            c.slice = p->D / cl;
            const int ncv = c.slice / 8;
            if (ncv > 512) return false;
            if (per_sm == 1) {
                c.b_vpt = ncv <= 256 ? 1 : 2;
            } else {
                // at most four consumer warps of two vectors: 160 threads at
                // ~166 registers, two CTAs in one SM's register file
                if (ncv > 256) return false;
                c.b_vpt = ncv <= 128 ? 1 : 2;
            }
            c.b_ncw = (ncv + 32 * c.b_vpt - 1) / (32 * c.b_vpt);
            c.b_per_sm = per_sm;
            c.b_slot_bytes = static_cast<int>(align_up(static_cast<uint32_t>(c.slice) * 2u, 128u));
            c.dy_slots = c.b_slot_bytes > 8192 ? 2 : 4;
            const long long budget = per_sm == 1 ? optin : optin / 2 - 1024;
            const long long csb = c.b_slot_bytes;
            const long long cfixed = make_cluster_layout(0, 1, c.b_slot_bytes, c.dy_slots, c.s_pad, cl).total + 64;
            const long long cavail = budget - cfixed;
            auto chunks_for = [&](int rows) {
                int k = 0;
                while (k < kMaxChunks &&
                       make_cluster_layout(k + 1, rows, c.b_slot_bytes, c.dy_slots, c.s_pad, cl).total <=
                           static_cast<uint32_t>(budget))
                    ++k;
                return k;
            };
            if (resident) {
                // a whole token per chunk when two fit, else quarters of a token (finer
                // releases let the next token's rows load during the write pass); the
                // slices stay with room for the next token to start loading
                c.b_rows = (2LL * S * csb <= cavail) ? S : (S + 3) / 4;
                c.b_chunks = chunks_for(c.b_rows);
                const int per_token = (S + c.b_rows - 1) / c.b_rows;
                if (c.b_chunks < (per_token == 1 ? 2 : per_token + (per_token + 1) / 2)) return false;
            } else {
                // at least four chunks in flight, at most 16 rows each, a
                // multiple of four rows when possible (the dot pass reduces
                // four rows at a time)
                long long g = cavail / (4 * csb);
                if (g > 16) g = 16;
                if (g >= 4) g &= ~3LL;
                if (g < 1) g = 1;
                c.b_rows = static_cast<int>(g);
                c.b_chunks = chunks_for(c.b_rows);
                if (c.b_chunks < 2) return false;
            }
            c.resident = resident ? 1 : 0;
            c.smem_bwd = make_cluster_layout(c.b_chunks, c.b_rows, c.b_slot_bytes, c.dy_slots, c.s_pad, cl).total;
            c.split = 1;  // the clusters' partial rows are always added by the finalize kernel
            const int active = bwd_cluster_max_active(c, p->R == p->D, p->out_norm != 0, S);
            if (active < 1) return false;
            long long ncl = active;
            if (p->N < ncl) ncl = p->N;
            if (!resident && cc.mode < 2 && cl < kClusterMax && ncl * token_bytes > dev.l2_bytes / 4 * 3)
                return false;  // a larger cluster shortens the reuse distance further
            c.nparts = static_cast<int>(ncl);
            c.grid = c.nparts * cl;
            *out = c;
            return true;
        };
        Plan c;
        bool found = false;
        if (cc.mode > 0) {
            found = try_cluster(cc.cl, cc.mode == 1, cc.mode == 3 ? 2 : 1, &c);
        } else {
            for (int cl = 2; cl <= kClusterMax && !found; cl *= 2) found = try_cluster(cl, false, 1, &c);
        }
        if (found) pl = c;
    }
    pl.ngroups = (pl.grid + kGroupTicket - 1) / kGroupTicket;
    const size_t W = static_cast<size_t>(p->R) + (p->out_norm ? static_cast<size_t>(p->D) : 0u);
    size_t off = align_up(static_cast<uint32_t>((pl.ngroups + 1) * 4), 256u);
    pl.ws_part_off = off;
    off += align_up(static_cast<uint32_t>(pl.nparts * W * 4), 256u);
    pl.ws_gpart_off = off;
    off += static_cast<size_t>(pl.ngroups) * W * 4;
    pl.ws_bytes = p->N == 0 ? 0 : off;
    *plan = pl;
    return ATTNRES_OK;
}

size_t align_up_sz(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Gradient rows: present, 16-byte aligned, disjoint from each other and from
// every source.
attnres_status check_dsrc(const attnres_params* p, void* const* dsrc, int64_t dsrc_ld) {
    if (dsrc_ld < p->D) return ATTNRES_ERR_INVALID_ARG;
    if (dsrc_ld % 8 != 0) return ATTNRES_ERR_ALIGNMENT;
    const size_t n_rows = static_cast<size_t>(p->N);
    const size_t d_bytes = n_rows == 0 ? 0 : ((n_rows - 1) * static_cast<size_t>(dsrc_ld) + p->D) * 2;
    const size_t s_bytes = n_rows == 0 ? 0 : ((n_rows - 1) * static_cast<size_t>(p->src_ld) + p->D) * 2;
    for (int s = 0; s < p->S; ++s) {
        if (!dsrc[s]) return ATTNRES_ERR_INVALID_ARG;
        if (!aligned16(dsrc[s])) return ATTNRES_ERR_ALIGNMENT;
    }
    for (int s = 0; s < p->S; ++s) {
        for (int t = 0; t < p->S; ++t) {
            if (t != s && ranges_overlap(dsrc[s], d_bytes, dsrc[t], d_bytes)) return ATTNRES_ERR_INVALID_ARG;
            if (ranges_overlap(dsrc[s], d_bytes, p->src[t], s_bytes)) return ATTNRES_ERR_INVALID_ARG;
        }
    }
    return ATTNRES_OK;
}

// ---------------------------------------------------------------- multi-query
attnres_status check_multi(const attnres_multi_params* p) {
    if (!p) return ATTNRES_ERR_INVALID_ARG;
    const attnres_status st = check_shape(&p->base);
    if (st != ATTNRES_OK) return st;
    if (p->M < 1 || p->M > ATTNRES_MAX_M) return ATTNRES_ERR_INVALID_ARG;
    if (p->base.out_norm) return ATTNRES_ERR_UNSUPPORTED;
    if (p->out_ld_m < 0 || p->out_ld_n < 0) return ATTNRES_ERR_INVALID_ARG;
    if (p->out_ld_m % 8 != 0 || p->out_ld_n % 8 != 0) return ATTNRES_ERR_ALIGNMENT;
    return ATTNRES_OK;
}

// Chunk ring for a resident token: the fewest chunks per token that leave
// room for one more chunk (so the next token starts loading), then as many
// chunks as fit; as a last resort the token alone.
template <typename F>
bool pick_ring(int S, F&& fits, int* rows, int* chunks) {
    for (int extra = 1; extra >= 0; --extra) {
        for (int cpt = 1; cpt <= S; ++cpt) {
            const int G = (S + cpt - 1) / cpt;
            if ((S + G - 1) / G != cpt) continue;
            if (!fits(cpt + extra, G)) continue;
            int K = cpt + extra;
            while (K < kMaxChunks && fits(K + 1, G)) ++K;
            *rows = G;
            *chunks = K;
            return true;
        }
    }
    return false;
}

// E > 0: per-token queries selected from an [E, R] bank (dq rows are bank rows).
attnres_status make_multi_plan(const attnres_multi_params* p, MultiPlan* plan, int E = 0) {
    DeviceInfo dev;
    if (!device_info(&dev)) return ATTNRES_ERR_CUDA;
    const attnres_params& b = p->base;
    MultiPlan pl{};
    pl.E = E;  // the occupancy queries below pick the kernels by it
    const int ncv = b.D / 8;
    const int M = p->M;
    pl.slot_bytes = static_cast<int>(align_up(static_cast<uint32_t>(b.D) * 2u, 128u));
    pl.s_pad = static_cast<int>(align_up(static_cast<uint32_t>(b.S), 4u));
    pl.m_pad = static_cast<int>(align_up(static_cast<uint32_t>(M), 4u));
    pl.kv0 = b.key_offset / 8;
    pl.nkv = (b.key_offset + b.R + 7) / 8 - pl.kv0;
    const uint32_t optin = static_cast<uint32_t>(dev.smem_optin);
    const long long sb = pl.slot_bytes;

    // Forward: as the single-query forward (two CTAs per SM when a thread owns
    // at most two vectors), with MB = 4 / (vectors per thread) queries per
    // pass over a token.  The queries stay in shared memory when they take at
    // most a quarter of it, else each block's MB queries are reloaded.
    pl.vpt = ncv <= 256 ? 1 : (ncv <= 512 ? 2 : 4);
    pl.ncw = (ncv + 32 * pl.vpt - 1) / (32 * pl.vpt);
    if (pl.ncw < 1 || pl.ncw > kMaxConsumerWarps) return ATTNRES_ERR_UNSUPPORTED;
    pl.mq = multi_fixed_m(M);
    pl.mb_f = multi_fwd_mb(M, pl.vpt);
    const int nblk = (M + pl.mb_f - 1) / pl.mb_f;
    bool fok = false;
    for (int cps = kMultiMaxCtasPerSm; cps >= 1 && !fok; --cps) {
        if (cps * (pl.ncw + 1) * 32 > 2048) continue;
        const uint32_t budget = cps > 1 ? optin / cps - 1024 : optin;
        const uint32_t qall = static_cast<uint32_t>(nblk * pl.mb_f) * static_cast<uint32_t>(pl.nkv) * 16u;
        int qrows = qall <= budget / 2 ? nblk * pl.mb_f : pl.mb_f;
        // selected queries: the whole bank (and a zero row for bad ids) when it
        // takes at most half the budget, else each block's rows per token
        const uint32_t ball = static_cast<uint32_t>(E + 1) * static_cast<uint32_t>(pl.nkv) * 16u;
        const int bank = (E > 0 && ball <= budget / 2) ? E + 1 : 0;
        if (E > 0) qrows = bank ? bank : pl.mb_f;
        auto ffits = [&](int chunks, int rows) {
            return make_multi_fwd_layout(chunks, rows, pl.slot_bytes, pl.s_pad, qrows, pl.nkv).total <= budget;
        };
        const long long fixed = make_multi_fwd_layout(0, 1, pl.slot_bytes, pl.s_pad, qrows, pl.nkv).total + 64;
        if (fixed + 2 * sb > budget) continue;
        long long gmax = (budget - fixed) / (2 * sb);
        if (gmax > kMaxGroup) gmax = kMaxGroup;
        if (gmax < 1) gmax = 1;
        const int groups = static_cast<int>((b.S + gmax - 1) / gmax);
        const int rows = (b.S + groups - 1) / groups;
        int chunks = 0;
        while (chunks < kMaxChunks && ffits(chunks + 1, rows)) ++chunks;
        if (chunks < 2) continue;
        int gc = chunks - 1;
        while (gc > 1 && gc * rows > kMaxGroup) --gc;
        pl.f_rows = rows;
        pl.f_chunks = chunks;
        pl.f_group = gc * rows;
        pl.qrows = qrows;
        pl.bank_f = bank;
        pl.smem_fwd = make_multi_fwd_layout(chunks, rows, pl.slot_bytes, pl.s_pad, qrows, pl.nkv).total;
        // more than one CTA per SM only when the kernel's registers allow it
        if (cps > 1 && multi_fwd_occupancy(pl) < cps) continue;
        long long fg = static_cast<long long>(cps) * dev.sm_count;
        if (b.N < fg) fg = b.N;
        pl.fgrid = static_cast<int>(fg < 1 ? 1 : fg);
        fok = true;
    }
    if (!fok) return ATTNRES_ERR_UNSUPPORTED;

    // Backward: a token's rows, its dy rows and the queries stay resident.
    pl.b_vpt = ncv <= 32 * kMultiBwdWarps ? 1 : 2;
    pl.b_ncw = (ncv + 32 * pl.b_vpt - 1) / (32 * pl.b_vpt);
    pl.mb_b = multi_bwd_mb(M, pl.b_vpt);
    const int nmb = (M + pl.mb_b - 1) / pl.mb_b;
    const bool dq_in_smem = nmb > 1;  // one block: dq in registers (selected: reduced into the workspace)
    const int dq_nkv = dq_in_smem ? pl.nkv : 0;
    const int dq_rows = E > 0 ? E : M;
    pl.bwd_ok = 0;
    int bcps = 1;
    // selected queries: first with the bank resident in shared memory, then
    // with each token's bank rows loaded per token
    for (int bank = (E > 0 && nmb == 1) ? E + 1 : 0; bank >= 0 && !pl.bwd_ok; bank = bank > 0 ? 0 : -1) {
        const int q_rows = bank > pl.m_pad ? bank : pl.m_pad;
        pl.bank_b = bank;
        for (int cps = kMultiMaxCtasPerSm; cps >= 1 && !pl.bwd_ok; --cps) {
            if (cps * (pl.b_ncw + 1) * 32 > 2048 || pl.b_ncw > kMultiBwdWarps) continue;
            const uint32_t budget = cps > 1 ? optin / cps - 1024 : optin;
            for (int ds = 2; ds >= 1 && !pl.bwd_ok; --ds) {
                auto bfits = [&](int K, int G) {
                    return make_multi_layout(K, G, pl.slot_bytes, M, ds, pl.s_pad, pl.m_pad, pl.nkv, dq_nkv, true,
                                             dq_rows, q_rows).total <= budget;
                };
                if (!pick_ring(b.S, bfits, &pl.b_rows, &pl.b_chunks)) continue;
                // the bank stays only where the ring still loads the next token meanwhile
                if (bank > 0 && pl.b_chunks < (b.S + pl.b_rows - 1) / pl.b_rows + 1) continue;
                pl.dy_slots = ds;
                pl.smem_bwd = make_multi_layout(pl.b_chunks, pl.b_rows, pl.slot_bytes, M, ds, pl.s_pad, pl.m_pad,
                                                pl.nkv, dq_nkv, true, dq_rows, q_rows).total;
                if (cps > 1 && multi_bwd_occupancy(pl) < cps) continue;
                pl.bwd_ok = 1;
                bcps = cps;
            }
        }
    }
    if (!pl.bwd_ok) pl.bank_b = 0;
    long long grid = static_cast<long long>(bcps) * dev.sm_count;
    if (b.N < grid) grid = b.N;
    pl.grid = static_cast<int>(grid < 1 ? 1 : grid);
    pl.ws_bytes = b.N == 0 ? 0 : static_cast<size_t>(pl.grid) * dq_rows * b.R * 4;

    // General backward (two kernels over column blocks, attnres_multi_general.cu):
    // every shape whose token does not fit the resident layout, and more than
    // kMultiResidentMaxM queries.
    // ATTNRES_MULTI_BWD=general / resident (read on every call) forces one
    // form where it fits, so both can be tested and timed on any shape.
    const char* form = std::getenv("ATTNRES_MULTI_BWD");
    const bool want_gen = form && std::strcmp(form, "general") == 0;
    const bool want_res = form && std::strcmp(form, "resident") == 0;
    pl.gen = 0;
    if (!pl.bwd_ok || (M > kMultiResidentMaxM && !want_res) || want_gen) {
        const int S = b.S;
        const int s8 = (S + 7) / 8 * 8;
        const int ntiles = s8 / 8;
        pl.gen_s8 = s8;
        pl.gen_kgroups = ntiles < kMultiCoefWarps ? kMultiCoefWarps / ntiles : 1;
        // coefficient table per source: alpha, b (queries padded to a multiple
        // of 4, for 16-byte loads) and c, padded to a multiple of 4 floats
        pl.gen_cs = 2 * ((M + 3) & ~3) + 4;
        // coefficient kernel: two CTAs per SM when their layouts fit in half of
        // it, each with a ring of at least two row blocks of the widest block
        // width that allows them (1024 columns down to 256, a multiple of 16
        // below that), holding as many buffers as fit.  Wide blocks first: the
        // copies are one 1-D bulk copy per row and block, and measured
        // (S=10, N=32768) 512-byte copies could not keep the SMs fed where
        // 1-2 KB ones could (M=16 D=1024: 1.28 ms at 256 columns, 1.04 at 512;
        // M=8 D=4096: 4.23 at 256, 3.30 at 1024).
        bool ok_a = false;
        int coef_ctas = 2;
        for (int pass = 0; pass < 4 && !ok_a; ++pass) {
            coef_ctas = pass < 2 ? 2 : 1;
            const size_t budget = coef_ctas == 2 ? optin / 2 - 1024 : optin;
            for (int dc = 1024; dc >= ((pass & 1) == 0 ? 256 : 16) && !ok_a; dc /= 2) {
                const int pitch = dc * 2 + 16;
                for (int bufs = kMultiGenMaxBufs; bufs >= 2; --bufs) {
                    const size_t sm = multi_gen_smem_a(bufs, s8, pitch, M, S, pl.gen_kgroups, pl.gen_cs);
                    if (sm > budget) continue;
                    ok_a = true;
                    pl.gen_dc = dc;
                    pl.gen_pitch = pitch;
                    pl.gen_bufs = bufs;
                    pl.gen_smem_a = sm;
                    break;  // the most buffers that fit at this width
                }
            }
        }
        // gradient kernel: 512 columns per column pair of a thread (two pairs
        // when the registers allow, M <= 8), source chunks of up to 8 rows, as
        // many token slots as leave the ring two tokens of rows; a bank of at
        // most 64 KB at these columns stays in shared memory
        const int pairs = (M <= 8 && b.D > kMultiGenColumns) ? 2 : 1;
        pl.gen_dcb = kMultiGenColumns * pairs;
        pl.gen_rows_b = S < 8 ? S : 8;
        pl.gen_bank_rows = (E > 0 && static_cast<long long>(E + 1) * pl.gen_dcb * 2 <= 65536) ? E + 1 : 0;
        const int per_token = (S + pl.gen_rows_b - 1) / pl.gen_rows_b;
        const int want_chunks = 2 * per_token < 16 ? (2 * per_token > 2 ? 2 * per_token : 2) : 16;
        bool ok_b = false;
        for (int ts = kMultiGenMaxSlots; ts >= 2 && !ok_b; --ts) {
            int chunks = 0;
            while (chunks < 16 && multi_gen_smem_b(S, pl.gen_cs, M, pl.gen_dcb, pl.gen_rows_b, chunks + 1,
                                                    pl.gen_bank_rows, ts) <= optin)
                ++chunks;
            if (chunks >= want_chunks || (ts == 2 && chunks >= 2)) {
                ok_b = true;
                pl.gen_tslots_b = ts;
                pl.gen_chunks_b = chunks;
                pl.gen_smem_b = multi_gen_smem_b(S, pl.gen_cs, M, pl.gen_dcb, pl.gen_rows_b, chunks,
                                                 pl.gen_bank_rows, ts);
            }
        }
        // the gradient kernel on the tensor cores (fixed queries, at most 16
        // sources: one 16-row MMA tile) with as many token slots as fit, from
        // kMultiGradMmaMinM queries up (its cost does not grow with the query
        // count, the SIMT kernel's does); ATTNRES_MULTI_GRAD=mma|simt (read on
        // every call) forces a form where it fits
        const char* gform = std::getenv("ATTNRES_MULTI_GRAD");
        const bool want_simt = gform && std::strcmp(gform, "simt") == 0;
        const bool want_mma = gform && std::strcmp(gform, "mma") == 0;
        pl.gen_grad_mma = 0;
        if (E == 0 && S <= 16 && !want_simt && (want_mma || M >= kMultiGradMmaMinM)) {
            for (int ts = kMultiGenMaxSlots; ts >= 2; --ts) {
                const size_t sm = multi_grad_mma_smem(S, pl.gen_cs, M, ts);
                if (sm <= optin) {
                    pl.gen_grad_mma = 1;
                    pl.gen_dcb = kMultiGenColumns;
                    pl.gen_tslots_b = ts;
                    pl.gen_smem_b = sm;
                    ok_b = true;
                    break;
                }
            }
        }
        if (ok_a && ok_b) {
            pl.gen = 1;
            pl.bwd_ok = 1;
            long long ga = static_cast<long long>(coef_ctas) * dev.sm_count;
            if (b.N < ga) ga = b.N;
            pl.gen_grid_a = static_cast<int>(ga < 1 ? 1 : ga);
            const int nbb = (b.D + pl.gen_dcb - 1) / pl.gen_dcb;
            long long groups = dev.sm_count / nbb;
            if (groups < 1) groups = 1;
            if (b.N < groups) groups = b.N;
            if (groups < 1) groups = 1;
            pl.gen_groups = static_cast<int>(groups);
            pl.gen_grid_b = pl.gen_groups * nbb;
            const size_t coef_bytes = static_cast<size_t>(b.N) * S * pl.gen_cs * 4;
            pl.gen_part_off = align_up_sz(coef_bytes, 256);
            pl.ws_bytes = b.N == 0 ? 0 : pl.gen_part_off + static_cast<size_t>(pl.gen_groups) * dq_rows * b.R * 4;
        }
    }
    *plan = pl;
    return ATTNRES_OK;
}

}  // namespace
}  // namespace attnres

using namespace attnres;

extern "C" {

const char* attnres_status_string(attnres_status s) {
    switch (s) {
        case ATTNRES_OK: return "ok";
        case ATTNRES_ERR_INVALID_ARG: return "invalid argument (size, flag or NULL pointer)";
        case ATTNRES_ERR_ALIGNMENT: return "alignment: rows must start on 16-byte boundaries, D and row strides multiples of 8";
        case ATTNRES_ERR_UNSUPPORTED: return "unsupported configuration for this build";
        case ATTNRES_ERR_WORKSPACE: return "workspace missing or too small";
        case ATTNRES_ERR_CUDA: return "CUDA runtime error";
        case ATTNRES_ERR_DEVICE: return "a kernel reported an error (a failed barrier wait or an out-of-range query id)";
        default: return "unknown status";
    }
}

attnres_status attnres_plan_info(const attnres_params* p, int64_t out[10]) {
    attnres_status st = check_shape(p);
    if (st != ATTNRES_OK) return st;
    if (!out) return ATTNRES_ERR_INVALID_ARG;
    Plan pl;
    st = make_plan(p, &pl);
    if (st != ATTNRES_OK) return st;
    out[0] = pl.grid;
    out[1] = pl.ncw * 1000 + pl.b_ncw;
    out[2] = pl.vpt * 1000 + pl.b_vpt;
    out[3] = pl.b_chunks * 1000 + pl.b_rows;
    out[4] = pl.f_chunks * 1000 + pl.f_rows;
    out[5] = pl.resident;
    out[6] = static_cast<int64_t>(pl.smem_bwd);
    out[7] = pl.split;
    out[8] = pl.cl;
    out[9] = pl.nparts;
    return ATTNRES_OK;
}

static attnres_status fwd_impl(const attnres_params* p, const void* q, const void* w_o, const void* delta,
                               int64_t delta_ld, void* partial_out, int64_t partial_ld, void* y, float* alpha,
                               float* rstd, float* logit, float* o_rstd, float* o_pre, void* stream,
                               long long test_withhold = 0, uint64_t test_wait_ns = 0) {
    attnres_status st = check_shape(p);
    if (st != ATTNRES_OK) return st;
    if (delta) {
        if (!partial_out) return ATTNRES_ERR_INVALID_ARG;
        if (delta_ld < p->D || partial_ld < p->D) return ATTNRES_ERR_INVALID_ARG;
        if (delta_ld % 8 != 0 || partial_ld % 8 != 0) return ATTNRES_ERR_ALIGNMENT;
    }
    if (p->N == 0) return ATTNRES_OK;
    if (delta && (!aligned16(delta) || !aligned16(partial_out))) return ATTNRES_ERR_ALIGNMENT;
    if (!q || !y || !alpha || !rstd || !logit) return ATTNRES_ERR_INVALID_ARG;
    if (p->out_norm && (!w_o || !o_rstd)) return ATTNRES_ERR_INVALID_ARG;
    if (!p->out_norm && o_pre) return ATTNRES_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned4(alpha) || !aligned4(rstd) || !aligned4(logit))
        return ATTNRES_ERR_ALIGNMENT;
    if (p->out_norm && !aligned4(o_rstd)) return ATTNRES_ERR_ALIGNMENT;
    if (o_pre && !aligned16(o_pre)) return ATTNRES_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(q) & 1u) || (w_o && (reinterpret_cast<uintptr_t>(w_o) & 1u)))
        return ATTNRES_ERR_ALIGNMENT;
    Plan pl;
    st = make_plan(p, &pl, delta != nullptr);
    if (st != ATTNRES_OK) return st;
    FwdArgs a;
    std::memset(&a, 0, sizeof a);
    for (int s = 0; s < p->S; ++s) a.src[s] = p->src[s];
    a.N = p->N;
    a.src_ld = p->src_ld;
    a.S = p->S;
    a.D = p->D;
    a.R = p->R;
    a.ko = p->key_offset;
    a.out_norm = p->out_norm;
    a.eps = p->eps;
    a.scale = p->scale;
    a.chunks = pl.f_chunks;
    a.rows = pl.f_rows;
    a.group = pl.f_group;
    a.slot_bytes = pl.slot_bytes;
    a.ncw = pl.ncw;
    a.s_pad = pl.s_pad;
    a.q = static_cast<const uint16_t*>(q);
    a.w_o = static_cast<const uint16_t*>(w_o);
    a.y = static_cast<uint16_t*>(y);
    a.alpha = alpha;
    a.rstd = rstd;
    a.logit = logit;
    a.o_rstd = o_rstd;
    a.o_pre = p->out_norm ? o_pre : nullptr;
    a.delta = static_cast<const uint16_t*>(delta);
    a.delta_ld = delta_ld;
    a.partial_out = static_cast<uint16_t*>(partial_out);
    a.partial_ld = partial_ld;
    a.test_withhold = test_withhold;
    a.test_wait_ns = test_wait_ns;
    return launch_fwd(pl, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTNRES_OK
                                                                              : ATTNRES_ERR_CUDA;
}

attnres_status attnres_fwd_withhold_for_test(const attnres_params* p, const void* q, const void* w_o, void* y,
                                             float* alpha, float* rstd, float* logit, float* o_rstd,
                                             int64_t withhold_fill, uint32_t wait_us, void* stream) {
    if (withhold_fill < 1 || wait_us < 1 || wait_us > 1000000u) return ATTNRES_ERR_INVALID_ARG;
    return fwd_impl(p, q, w_o, nullptr, 0, nullptr, 0, y, alpha, rstd, logit, o_rstd, nullptr, stream,
                    withhold_fill, static_cast<uint64_t>(wait_us) * 1000ull);
}

attnres_status attnres_fwd(const attnres_params* p, const void* q, const void* w_o, void* y,
                           float* alpha, float* rstd, float* logit, float* o_rstd, float* o_pre,
                           void* stream) {
    return fwd_impl(p, q, w_o, nullptr, 0, nullptr, 0, y, alpha, rstd, logit, o_rstd, o_pre, stream);
}

attnres_status attnres_fwd_partial(const attnres_params* p, const void* q, const void* w_o,
                                   const void* delta, int64_t delta_ld, void* partial_out,
                                   int64_t partial_ld, void* y, float* alpha, float* rstd,
                                   float* logit, float* o_rstd, float* o_pre, void* stream) {
    if (!delta && p && p->N > 0) return ATTNRES_ERR_INVALID_ARG;
    if (!delta) return check_shape(p);
    return fwd_impl(p, q, w_o, delta, delta_ld, partial_out, partial_ld, y, alpha, rstd, logit, o_rstd, o_pre,
                    stream);
}

size_t attnres_bwd_workspace_bytes(const attnres_params* p) {
    if (check_shape(p) != ATTNRES_OK) return 0;
    Plan pl;
    if (make_plan(p, &pl) != ATTNRES_OK) return 0;
    return pl.ws_bytes;
}

static attnres_status bwd_impl(const attnres_params* p, const void* q, const void* w_o, const void* dy,
                               const float* alpha, const float* rstd, const float* logit,
                               const float* o_rstd, const float* o_pre, const void* g_last, int64_t g_ld,
                               void* const* dsrc, int64_t dsrc_ld, void* dq, float* dq_f32, void* dw_o,
                               float* dw_o_f32, void* workspace, size_t workspace_bytes, void* stream) {
    attnres_status st = check_shape(p);
    if (g_last && (g_ld < p->D)) return ATTNRES_ERR_INVALID_ARG;
    if (g_last && (g_ld % 8 != 0 || !aligned16(g_last))) return ATTNRES_ERR_ALIGNMENT;
    if (st != ATTNRES_OK) return st;
    if (p->N == 0) {
        // Empty sums: dq and dw_o are zero; nothing else is touched.
        if (!dq || (p->out_norm && !dw_o)) return ATTNRES_ERR_INVALID_ARG;
        cudaStream_t s0 = static_cast<cudaStream_t>(stream);
        if (cudaMemsetAsync(dq, 0, static_cast<size_t>(p->R) * 2, s0) != cudaSuccess ||
            (dq_f32 && cudaMemsetAsync(dq_f32, 0, static_cast<size_t>(p->R) * 4, s0) != cudaSuccess) ||
            (dw_o && cudaMemsetAsync(dw_o, 0, static_cast<size_t>(p->D) * 2, s0) != cudaSuccess) ||
            (dw_o_f32 && cudaMemsetAsync(dw_o_f32, 0, static_cast<size_t>(p->D) * 4, s0) != cudaSuccess))
            return ATTNRES_ERR_CUDA;
        return ATTNRES_OK;
    }
    if (!q || !dy || !alpha || !rstd || !logit || !dsrc || !dq) return ATTNRES_ERR_INVALID_ARG;
    if (p->out_norm && (!w_o || !o_rstd || !dw_o)) return ATTNRES_ERR_INVALID_ARG;
    if (!p->out_norm && o_pre) return ATTNRES_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned4(alpha) || !aligned4(rstd) || !aligned4(logit))
        return ATTNRES_ERR_ALIGNMENT;
    if (p->out_norm && !aligned4(o_rstd)) return ATTNRES_ERR_ALIGNMENT;
    if (o_pre && !aligned16(o_pre)) return ATTNRES_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(q) & 1u) || (reinterpret_cast<uintptr_t>(dq) & 1u) ||
        (dq_f32 && !aligned4(dq_f32)) || (dw_o && (reinterpret_cast<uintptr_t>(dw_o) & 1u)) ||
        (dw_o_f32 && !aligned4(dw_o_f32)) || (w_o && (reinterpret_cast<uintptr_t>(w_o) & 1u)))
        return ATTNRES_ERR_ALIGNMENT;
    st = check_dsrc(p, dsrc, dsrc_ld);
    if (st != ATTNRES_OK) return st;
    Plan pl;
    st = make_plan(p, &pl, false, g_last != nullptr);
    if (st != ATTNRES_OK) return st;
    if (!workspace || workspace_bytes < pl.ws_bytes) return ATTNRES_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTNRES_ERR_ALIGNMENT;
    BwdArgs a;
    std::memset(&a, 0, sizeof a);
    for (int s = 0; s < p->S; ++s) {
        a.src[s] = p->src[s];
        a.dsrc[s] = dsrc[s];
    }
    a.N = p->N;
    a.src_ld = p->src_ld;
    a.dsrc_ld = dsrc_ld;
    {
        // evenly spaced output rows (a packed [S, N, D] gradient) let the
        // kernel step from one source's row to the next with one add
        const long long st = p->S > 1 ? static_cast<long long>(reinterpret_cast<uintptr_t>(dsrc[1])) -
                                            static_cast<long long>(reinterpret_cast<uintptr_t>(dsrc[0]))
                                      : 0;
        bool even = p->S > 1 && st != 0;
        for (int s2 = 2; even && s2 < p->S; ++s2)
            even = static_cast<long long>(reinterpret_cast<uintptr_t>(dsrc[s2])) -
                       static_cast<long long>(reinterpret_cast<uintptr_t>(dsrc[s2 - 1])) == st;
        a.dsrc_stride = even ? st : 0;
    }
    a.S = p->S;
    a.D = p->D;
    a.R = p->R;
    a.ko = p->key_offset;
    a.out_norm = p->out_norm;
    a.eps = p->eps;
    a.scale = p->scale;
    a.chunks = pl.b_chunks;
    a.rows = pl.b_rows;
    a.dy_slots = pl.dy_slots;
    a.slot_bytes = pl.b_slot_bytes;
    a.ncw = pl.b_ncw;
    a.s_pad = pl.s_pad;
    a.resident = pl.resident;
    a.split = pl.split;
    a.ngroups = pl.ngroups;
    a.cl = pl.cl;
    a.slice = pl.slice;
    a.q = static_cast<const uint16_t*>(q);
    a.w_o = static_cast<const uint16_t*>(w_o);
    a.dy = static_cast<const uint16_t*>(dy);
    a.alpha = alpha;
    a.rstd = rstd;
    a.logit = logit;
    a.o_rstd = o_rstd;
    a.o_pre = o_pre;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    a.tickets = reinterpret_cast<unsigned*>(ws);
    a.part = reinterpret_cast<float*>(ws + pl.ws_part_off);
    a.part_rows = pl.nparts;
    a.gpart = reinterpret_cast<float*>(ws + pl.ws_gpart_off);
    a.dq = static_cast<uint16_t*>(dq);
    a.dq_f32 = dq_f32;
    a.dw_o = static_cast<uint16_t*>(dw_o);
    a.dw_o_f32 = dw_o_f32;
    a.dlast_add = static_cast<const uint16_t*>(g_last);
    a.dlast_add_ld = g_ld;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!pl.split) {
        if (cudaMemsetAsync(a.tickets, 0, static_cast<size_t>(pl.ngroups + 1) * 4, s) != cudaSuccess)
            return ATTNRES_ERR_CUDA;
    }
    return launch_bwd(pl, a, s) == cudaSuccess ? ATTNRES_OK : ATTNRES_ERR_CUDA;
}

attnres_status attnres_bwd(const attnres_params* p, const void* q, const void* w_o, const void* dy,
                           const float* alpha, const float* rstd, const float* logit,
                           const float* o_rstd, const float* o_pre, void* const* dsrc,
                           int64_t dsrc_ld, void* dq, float* dq_f32, void* dw_o, float* dw_o_f32,
                           void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(p, q, w_o, dy, alpha, rstd, logit, o_rstd, o_pre, nullptr, 0, dsrc, dsrc_ld, dq, dq_f32,
                    dw_o, dw_o_f32, workspace, workspace_bytes, stream);
}

attnres_status attnres_bwd_partial(const attnres_params* p, const void* q, const void* w_o, const void* dy,
                                   const float* alpha, const float* rstd, const float* logit,
                                   const float* o_rstd, const float* o_pre, const void* g_partial,
                                   int64_t g_ld, void* const* dsrc, int64_t dsrc_ld, void* dq,
                                   float* dq_f32, void* dw_o, float* dw_o_f32, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    return bwd_impl(p, q, w_o, dy, alpha, rstd, logit, o_rstd, o_pre, g_partial, g_ld, dsrc, dsrc_ld, dq,
                    dq_f32, dw_o, dw_o_f32, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Backward without a caller workspace.  Its scratch is this file-scope device
// array; host code must not use the name as an address (on the host it is a
// stand-in), so each device's address is looked up once with cudaGetSymbolAddress
// and handed to attnres_bwd as the workspace.  The tickets that must start at
// zero are cleared on the caller's stream by attnres_bwd itself.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTNRES_NOALLOC_SCRATCH_BYTES];

static void* noalloc_scratch_address(int dev) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = ptr;
    }
    return addr[dev];
}

attnres_status attnres_bwd_noalloc(const attnres_params* p, const void* q, const void* w_o,
                                   const void* dy, const float* alpha, const float* rstd,
                                   const float* logit, const float* o_rstd, const float* o_pre,
                                   void* const* dsrc, int64_t dsrc_ld, void* dq, float* dq_f32,
                                   void* dw_o, float* dw_o_f32, void* stream) {
    attnres_status st = check_shape(p);
    if (st != ATTNRES_OK) return st;
    const size_t need = attnres_bwd_workspace_bytes(p);
    if (need > ATTNRES_NOALLOC_SCRATCH_BYTES) return ATTNRES_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTNRES_ERR_CUDA;
    void* scratch = noalloc_scratch_address(dev);
    if (!scratch) return ATTNRES_ERR_CUDA;
    return attnres_bwd(p, q, w_o, dy, alpha, rstd, logit, o_rstd, o_pre, dsrc, dsrc_ld, dq, dq_f32,
                       dw_o, dw_o_f32, scratch, ATTNRES_NOALLOC_SCRATCH_BYTES, stream);
}

attnres_status attnres_check_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTNRES_ERR_CUDA;
    const unsigned f = take_fwd_error();
    const unsigned b = take_bwd_error();
    const unsigned mf = take_multi_fwd_error();
    const unsigned mb = take_multi_bwd_error();
    const unsigned mg = take_multi_gen_error();
    const unsigned mm = take_multi_mma_error();
    const unsigned mg2 = take_multi_grad_mma_error();
    if (f == 0xffffffffu || b == 0xffffffffu || mf == 0xffffffffu || mb == 0xffffffffu || mg == 0xffffffffu ||
        mm == 0xffffffffu || mg2 == 0xffffffffu)
        return ATTNRES_ERR_CUDA;
    return (f || b || mf || mb || mg || mm || mg2) ? ATTNRES_ERR_DEVICE : ATTNRES_OK;
}

// ---------------------------------------------------------------------------
// Multi-query read.
// ---------------------------------------------------------------------------
int attnres_jit_kernel_count(void) { return jit_fwd_kernels(); }

int attnres_multi_fwd_tensor_cores(const attnres_multi_params* p, int32_t E) {
    if (check_multi(p) != ATTNRES_OK) return -1;
    DeviceInfo dev;
    if (!device_info(&dev)) return -1;
    MmaPlan mp;
    return plan_multi_fwd_mma(p, E > 0 ? E : 0, dev.sm_count, dev.smem_optin, &mp) ? 1 : 0;
}

int attnres_debug_checks(void) {
#ifdef ATTNRES_DEBUG
    return 1;
#else
    return 0;
#endif
}

attnres_status attnres_multi_plan_info(const attnres_multi_params* p, int64_t out[10]) {
    attnres_status st = check_multi(p);
    if (st != ATTNRES_OK) return st;
    if (!out) return ATTNRES_ERR_INVALID_ARG;
    MultiPlan pl;
    st = make_multi_plan(p, &pl);
    if (st != ATTNRES_OK) return st;
    if (!pl.bwd_ok) return ATTNRES_ERR_UNSUPPORTED;
    out[0] = static_cast<int64_t>(pl.fgrid) * 1000 + pl.grid;
    out[1] = pl.ncw * 1000 + pl.b_ncw;
    out[2] = pl.vpt * 1000 + pl.b_vpt;
    out[3] = pl.mb_f * 1000 + pl.mb_b;
    out[4] = pl.f_chunks * 1000 + pl.f_rows;
    out[5] = pl.b_chunks * 1000 + pl.b_rows;
    out[6] = pl.dy_slots;
    out[7] = static_cast<int64_t>(pl.gen ? pl.gen_smem_b : pl.smem_bwd);
    out[8] = pl.gen ? 1 + pl.gen_grad_mma : 0;
    out[9] = pl.gen ? pl.gen_groups : 0;
    return ATTNRES_OK;
}

static attnres_status multi_fwd_impl(const attnres_multi_params* p, const void* q, int E, const int64_t* ids,
                                     void* y, float* alpha, float* rstd, float* logit, void* stream) {
    attnres_status st = check_multi(p);
    if (st != ATTNRES_OK) return st;
    const attnres_params& b = p->base;
    if (ids && E < 1) return ATTNRES_ERR_INVALID_ARG;
    if (b.N == 0) return ATTNRES_OK;
    if (!q || !y || !alpha || !rstd || !logit) return ATTNRES_ERR_INVALID_ARG;
    if (ids && (reinterpret_cast<uintptr_t>(ids) & 7u)) return ATTNRES_ERR_ALIGNMENT;
    if (!aligned16(y) || !aligned4(alpha) || !aligned4(rstd) || !aligned4(logit) ||
        (reinterpret_cast<uintptr_t>(q) & 1u))
        return ATTNRES_ERR_ALIGNMENT;
    MultiPlan pl;
    st = make_multi_plan(p, &pl, ids ? E : 0);
    if (st != ATTNRES_OK) return st;
    MultiFwdArgs a;
    std::memset(&a, 0, sizeof a);
    for (int s = 0; s < b.S; ++s) a.src[s] = b.src[s];
    a.N = b.N;
    a.src_ld = b.src_ld;
    a.y_ms = p->out_ld_m;
    a.y_ns = p->out_ld_n;
    a.S = b.S;
    a.D = b.D;
    a.R = b.R;
    a.ko = b.key_offset;
    a.M = p->M;
    a.eps = b.eps;
    a.scale = b.scale;
    a.chunks = pl.f_chunks;
    a.rows = pl.f_rows;
    a.group = pl.f_group;
    a.qrows = pl.qrows;
    a.slot_bytes = pl.slot_bytes;
    a.ncw = pl.ncw;
    a.s_pad = pl.s_pad;
    a.kv0 = pl.kv0;
    a.nkv = pl.nkv;
    a.q = static_cast<const uint16_t*>(q);
    a.ids = reinterpret_cast<const long long*>(ids);
    a.E = ids ? E : 0;
    a.bank_rows = ids ? pl.bank_f : 0;
    a.y = static_cast<uint16_t*>(y);
    a.alpha = alpha;
    a.rstd = rstd;
    a.logit = logit;
    // several queries over tokens that fit in shared memory: the tensor-core form
    DeviceInfo dev;
    MmaPlan mp;
    if (device_info(&dev) && plan_multi_fwd_mma(p, ids ? E : 0, dev.sm_count, dev.smem_optin, &mp))
        return launch_multi_fwd_mma(mp, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTNRES_OK
                                                                                             : ATTNRES_ERR_CUDA;
    return launch_multi_fwd(pl, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTNRES_OK
                                                                                    : ATTNRES_ERR_CUDA;
}

attnres_status attnres_multi_fwd(const attnres_multi_params* p, const void* q, void* y, float* alpha,
                                 float* rstd, float* logit, void* stream) {
    return multi_fwd_impl(p, q, 0, nullptr, y, alpha, rstd, logit, stream);
}

attnres_status attnres_selected_fwd(const attnres_multi_params* p, const void* bank, int32_t E,
                                    const int64_t* ids, void* y, float* alpha, float* rstd, float* logit,
                                    void* stream) {
    if (E < 1 || (p && p->base.N > 0 && !ids)) return ATTNRES_ERR_INVALID_ARG;
    return multi_fwd_impl(p, bank, E, ids, y, alpha, rstd, logit, stream);
}

static size_t multi_ws_impl(const attnres_multi_params* p, int E) {
    if (check_multi(p) != ATTNRES_OK) return 0;
    MultiPlan pl;
    if (make_multi_plan(p, &pl, E) != ATTNRES_OK) return 0;
    return pl.ws_bytes;
}

size_t attnres_multi_bwd_workspace_bytes(const attnres_multi_params* p) { return multi_ws_impl(p, 0); }

size_t attnres_selected_bwd_workspace_bytes(const attnres_multi_params* p, int32_t E) {
    return E < 1 ? 0 : multi_ws_impl(p, E);
}

static attnres_status multi_bwd_impl(const attnres_multi_params* p, const void* q, int E, const int64_t* ids,
                                     const void* dy, const float* alpha, const float* rstd, const float* logit,
                                     void* const* dsrc, int64_t dsrc_ld, void* dq, float* dq_f32,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    attnres_status st = check_multi(p);
    if (st != ATTNRES_OK) return st;
    const attnres_params& b = p->base;
    cudaStream_t s0 = static_cast<cudaStream_t>(stream);
    const size_t nq = static_cast<size_t>(ids ? E : p->M) * static_cast<size_t>(b.R);
    if (ids && (reinterpret_cast<uintptr_t>(ids) & 7u)) return ATTNRES_ERR_ALIGNMENT;
    if (!dq) return ATTNRES_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(dq) & 1u) || (dq_f32 && !aligned4(dq_f32))) return ATTNRES_ERR_ALIGNMENT;
    if (b.N == 0) {
        if (cudaMemsetAsync(dq, 0, nq * 2, s0) != cudaSuccess ||
            (dq_f32 && cudaMemsetAsync(dq_f32, 0, nq * 4, s0) != cudaSuccess))
            return ATTNRES_ERR_CUDA;
        return ATTNRES_OK;
    }
    if (!q || !dy || !alpha || !rstd || !logit || !dsrc) return ATTNRES_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned4(alpha) || !aligned4(rstd) || !aligned4(logit) ||
        (reinterpret_cast<uintptr_t>(q) & 1u))
        return ATTNRES_ERR_ALIGNMENT;
    st = check_dsrc(&b, dsrc, dsrc_ld);
    if (st != ATTNRES_OK) return st;
    MultiPlan pl;
    st = make_multi_plan(p, &pl, ids ? E : 0);
    if (st != ATTNRES_OK) return st;
    if (!pl.bwd_ok) return ATTNRES_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < pl.ws_bytes) return ATTNRES_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTNRES_ERR_ALIGNMENT;
    if (pl.gen) {
        MultiGenArgs g;
        std::memset(&g, 0, sizeof g);
        for (int s = 0; s < b.S; ++s) {
            g.src[s] = b.src[s];
            g.dsrc[s] = dsrc[s];
        }
        g.N = b.N;
        g.src_ld = b.src_ld;
        g.dsrc_ld = dsrc_ld;
        g.dy_ms = p->out_ld_m;
        g.dy_ns = p->out_ld_n;
        g.S = b.S;
        g.D = b.D;
        g.R = b.R;
        g.ko = b.key_offset;
        g.M = p->M;
        g.E = ids ? E : 0;
        g.scale = b.scale;
        g.s8 = pl.gen_s8;
        g.kgroups = pl.gen_kgroups;
        g.bufs = pl.gen_bufs;
        g.dc = pl.gen_dc;
        g.nblocks = (b.D + pl.gen_dc - 1) / pl.gen_dc;
        g.pitch = pl.gen_pitch;
        g.cs = pl.gen_cs;
        g.dcb = pl.gen_dcb;
        g.rows_b = pl.gen_rows_b;
        g.chunks_b = pl.gen_chunks_b;
        g.bank_rows = ids ? pl.gen_bank_rows : 0;
        g.tslots_b = pl.gen_tslots_b;
        g.q = static_cast<const uint16_t*>(q);
        g.ids = reinterpret_cast<const long long*>(ids);
        g.dy = static_cast<const uint16_t*>(dy);
        g.alpha = alpha;
        g.rstd = rstd;
        g.logit = logit;
        unsigned char* ws = static_cast<unsigned char*>(workspace);
        g.coef = reinterpret_cast<float*>(ws);
        g.part = reinterpret_cast<float*>(ws + pl.gen_part_off);
        g.dq = static_cast<uint16_t*>(dq);
        g.dq_f32 = dq_f32;
        return launch_multi_bwd_general(pl, g, s0) == cudaSuccess ? ATTNRES_OK : ATTNRES_ERR_CUDA;
    }
    MultiBwdArgs a;
    std::memset(&a, 0, sizeof a);
    for (int s = 0; s < b.S; ++s) {
        a.src[s] = b.src[s];
        a.dsrc[s] = dsrc[s];
    }
    a.N = b.N;
    a.src_ld = b.src_ld;
    a.dsrc_ld = dsrc_ld;
    a.dy_ms = p->out_ld_m;
    a.dy_ns = p->out_ld_n;
    a.S = b.S;
    a.D = b.D;
    a.R = b.R;
    a.ko = b.key_offset;
    a.M = p->M;
    a.eps = b.eps;
    a.scale = b.scale;
    a.chunks = pl.b_chunks;
    a.rows = pl.b_rows;
    a.slot_bytes = pl.slot_bytes;
    a.dy_slots = pl.dy_slots;
    a.ncw = pl.b_ncw;
    a.s_pad = pl.s_pad;
    a.m_pad = pl.m_pad;
    a.kv0 = pl.kv0;
    a.nkv = pl.nkv;
    a.q = static_cast<const uint16_t*>(q);
    a.dy = static_cast<const uint16_t*>(dy);
    a.alpha = alpha;
    a.rstd = rstd;
    a.logit = logit;
    a.part = static_cast<float*>(workspace);
    a.dq = static_cast<uint16_t*>(dq);
    a.dq_f32 = dq_f32;
    a.ids = reinterpret_cast<const long long*>(ids);
    a.E = ids ? E : 0;
    a.bank_rows = ids ? pl.bank_b : 0;
    return launch_multi_bwd(pl, a, s0) == cudaSuccess ? ATTNRES_OK : ATTNRES_ERR_CUDA;
}

attnres_status attnres_multi_bwd(const attnres_multi_params* p, const void* q, const void* dy,
                                 const float* alpha, const float* rstd, const float* logit,
                                 void* const* dsrc, int64_t dsrc_ld, void* dq, float* dq_f32,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    return multi_bwd_impl(p, q, 0, nullptr, dy, alpha, rstd, logit, dsrc, dsrc_ld, dq, dq_f32, workspace,
                          workspace_bytes, stream);
}

attnres_status attnres_selected_bwd(const attnres_multi_params* p, const void* bank, int32_t E,
                                    const int64_t* ids, const void* dy, const float* alpha,
                                    const float* rstd, const float* logit, void* const* dsrc,
                                    int64_t dsrc_ld, void* dbank, float* dbank_f32, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    if (E < 1 || (p && p->base.N > 0 && !ids)) return ATTNRES_ERR_INVALID_ARG;
    if (!ids) {  // no tokens: the bank gradient is zero
        attnres_status st = check_multi(p);
        if (st != ATTNRES_OK) return st;
        if (!dbank) return ATTNRES_ERR_INVALID_ARG;
        const size_t nb = static_cast<size_t>(E) * static_cast<size_t>(p->base.R);
        cudaStream_t s0 = static_cast<cudaStream_t>(stream);
        if (cudaMemsetAsync(dbank, 0, nb * 2, s0) != cudaSuccess ||
            (dbank_f32 && cudaMemsetAsync(dbank_f32, 0, nb * 4, s0) != cudaSuccess))
            return ATTNRES_ERR_CUDA;
        return ATTNRES_OK;
    }
    return multi_bwd_impl(p, bank, E, ids, dy, alpha, rstd, logit, dsrc, dsrc_ld, dbank, dbank_f32, workspace,
                          workspace_bytes, stream);
}

}  // extern "C"
