// gemm.cu - the draft FC (2h -> h, bias) and the shared LM head (h -> V) as streamed-weight GEMMs.
//
// EAGLE notes ch. 04 §4.1 / zdszero "draft 结构": f^ = FC([f || e(t)]) and z = LM_head(f^).  At
// draft time the rows (frontier nodes) are few (1..256) and the weights are large (64 MiB to
// 1 GB), so every launch streams its weight matrix through shared memory exactly once:
//
//   swap-AB     the weight tile is the MMA's A operand (M = 128 weight rows) and the activation
//               rows are its N (16..256), so one weight byte feeds all rows of the batch;
//   TMA         a producer warp streams 128x64 bf16 weight tiles (16 KB, 128-byte swizzle) and
//               the matching 64-wide slice of the activation rows into a ring of stages;
//   tcgen05     one thread issues tcgen05.mma (kind::f16, bf16 in, fp32 accumulate) into a
//               double-buffered TMEM accumulator; tcgen05.commit frees each stage;
//   epilogue    four warps read the accumulator with tcgen05.ld (one TMEM lane per weight row)
//               and write Y[r][o] coalesced along o (+ bias, rounding to bf16 for the FC);
//   stream-K    all k-blocks of all tiles are one sequence split evenly over one CTA per SM, so
//               every SM streams the same number of weight bytes whatever the tile count; a tile
//               cut between CTAs is summed in ascending CTA order, so results are deterministic:
//               up to 16 rows by the last CTA to arrive (atomic ticket, no waiting); above, when
//               every CTA covers a whole tile, by the CTA that reaches the tile at the end of its
//               range and finds its partner's ticket in (the partner's partial bulk-copied into
//               its idle ring, its own values straight from TMEM), else by a second launch;
//   bulk stores above 16 rows every 32-row group of outputs or partials is assembled in shared
//               memory and leaves by one bulk store (TMA tensor store into Y, 1-D bulk store of
//               partials) instead of per-thread stores to rows far apart;
//   CTA pairs   above 16 rows, with an even number of weight tiles, the CTAs run as
//               pairs (clusters of 2) on tcgen05 with .cta_group::2: one MMA of M = 256 covers
//               the pair's two adjacent weight tiles, each CTA streams its own tile's weights and
//               half of the activation rows, and the MMA reads both halves from the two CTAs'
//               shared memory.  An activation byte brought into an SM then feeds 256 weight rows
//               instead of 128: per k-block an SM takes in 16 KB of weights and n/2 x 128 B of
//               activations (32 KB at 256 rows, against 48 KB).  The stream-K split is over pairs
//               (k-blocks of pair tiles), and each CTA sums and writes its own tile as before;
//   row chunks  more rows than one MMA's N (256) are taken in chunks of 256: a unit of the split
//               is (weight tile or pair, row chunk), weight-major, so a worker runs the chunks of
//               one weight tile back to back (its later passes find the tile in L2) and the
//               whole product is one launch (the draft decoder layer's projections over every
//               node of a batch of trees).
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace eagle {
namespace {

constexpr int BM = kLinearTileM;
constexpr int BK = kLinearTileK;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB weight tile
constexpr int kMaxStages = 16;
constexpr int kThreads = 192;  // warp 0: TMA producer, warp 1: MMA issuer, warps 2-5: epilogue
constexpr size_t kMaxDynSmem = 232448;  // 227 KB per CTA on sm_100-class parts
constexpr int kGroupRows = 32;  // rows of one bulk-stored group of outputs or partials
constexpr uint32_t kGroupBytes = kGroupRows * BM * 4u;  // one group of a 128-wide tile in fp32
constexpr uint32_t kOutStageBytes = 2u * kGroupBytes;  // two staging buffers for bulk stores

struct SmemCtl {
    uint64_t full[kMaxStages];   // TMA -> MMA: stage loaded
    uint64_t empty[kMaxStages];  // MMA -> TMA: stage consumed
    uint64_t acc_full[2];        // MMA -> epilogue: accumulator ready
    uint64_t acc_empty[2];       // epilogue -> MMA: accumulator drained (4 warps arrive)
    uint64_t fix;                // split-tile owner: the other CTA's partial staged in the ring
    uint64_t drain;              // used only when unwinding after a timeout
    uint32_t tmem_base;
    int32_t abort;
    int32_t is_last;
    int32_t fix_chunks;          // staged copies issued on `fix` (phases), for unwinding
};

struct LinearArgs {
    int32_t M, K, rows, n_tile, num_kb, num_tiles, stages, tmem_cols;
    const __nv_bfloat16 *bias;
    void *out;
    int64_t ldo;
    int32_t out_bf16;
    int32_t defer;  // split tiles: write partials only; linear_reduce_kernel sums them
    int32_t owner_fix;  // split tiles summed in the launch by the CTA that finds its partner done
    int32_t pair;       // 1: CTA pairs (.cta_group::2), the stream-K split over pairs of tiles
    int32_t slots;      // partial-sum slots of the launch: two per CTA of the main kernel
    int32_t num_wtiles; // weight units: tiles, or pairs of tiles
    int32_t num_chunks; // row chunks of n_tile rows; the split's units are (weight unit, chunk)
    int32_t y_tma;      // 32-row groups of Y and of partials go out by bulk stores (tmap_y valid)
    int32_t out_stage_bytes;  // shared-memory staging of those groups (after the ring)
    float *partials;
    int32_t *counters;
    int32_t *status;
};

// a / b for a >= 0, b > 0: one 32-bit division when a fits in 32 bits (64-bit division is a
// long software sequence).
__device__ __forceinline__ int64_t div_nonneg(int64_t a, int64_t b) {
    if ((static_cast<uint64_t>(a) >> 32) == 0 && (static_cast<uint64_t>(b) >> 32) == 0)
        return static_cast<uint32_t>(a) / static_cast<uint32_t>(b);
    return a / b;
}

// Worker (CTA, or CTA pair) whose k-block range [total*g/G, total*(g+1)/G) contains k-block p.
__device__ __forceinline__ int32_t cta_of(int64_t p, int64_t total, int32_t G) {
    return static_cast<int32_t>(div_nonneg((p + 1) * G + total - 1, total)) - 1;
}

// A worker's partial sums of one of its (at most two) split tiles: slot 0 for the tile its range
// starts in, 1 for the one it ends in; with CTA pairs each CTA of the pair (rank) has its own.
__device__ __forceinline__ float *part_slot(const LinearArgs &a, int32_t worker, int32_t slot, int32_t rank) {
    int32_t i = ((worker * 2 + slot) << a.pair) + rank;
    if (!dcheck(i >= 0 && i < a.slots, a.status)) i = 0;
    return a.partials + static_cast<size_t>(i) * a.n_tile * BM;
}

__device__ __forceinline__ void store_y(const LinearArgs &a, int32_t r, int32_t o, float v) {
    if (a.out_bf16)
        reinterpret_cast<__nv_bfloat16 *>(a.out)[static_cast<int64_t>(r) * a.ldo + o] =
            __float2bfloat16_rn(v);
    else
        reinterpret_cast<float *>(a.out)[static_cast<int64_t>(r) * a.ldo + o] = v;
}

// Writes rows n0 .. n0 + 31 of this thread's column (m_local) of a 128-wide tile through one of two
// shared-memory staging buffers; thread et 0 sends the group with one bulk store: a TMA tensor
// store into Y (to_y: rows and columns outside Y are dropped; bf16 when Y is bf16) or a 1-D bulk
// store of the rows into the partial slot `part` (fp32, [row][128]).  All 128 epilogue threads.
__device__ __forceinline__ void group_store(const LinearArgs &a, const CUtensorMap *tmap_y, uint8_t *out_stage,
                                            int32_t &gi, int32_t et, int32_t m_local, const float (&v)[kGroupRows],
                                            bool to_y, float *part, int32_t tile, int32_t n0, int32_t row0,
                                            int32_t rows_c) {
    uint8_t *buf = out_stage + static_cast<size_t>(gi & 1) * kGroupBytes;
    if (et == 0 && gi >= 2) bulk_wait_read<1>();  // the store of group gi - 2 has read buf
    named_barrier_sync(1, 128);
    if (to_y && a.out_bf16) {
        __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(buf);
#pragma unroll
        for (int j = 0; j < kGroupRows; ++j) ob[j * BM + m_local] = __float2bfloat16_rn(v[j]);
    } else {
        float *ob = reinterpret_cast<float *>(buf);
#pragma unroll
        for (int j = 0; j < kGroupRows; ++j) ob[j * BM + m_local] = v[j];
    }
    fence_proxy_async_smem();  // the writes above, before the bulk store reads them
    named_barrier_sync(1, 128);
    if (et == 0) {
        if (to_y)
            tma_store_2d(tmap_y, buf, tile * BM, row0 + n0);
        else
            bulk_store(part + static_cast<size_t>(n0) * BM, buf,
                       static_cast<uint32_t>(min(kGroupRows, rows_c - n0)) * BM * 4u);
        bulk_commit();
    }
    ++gi;
}

// Sums a split tile's partials in ascending CTA order (the order of every other path) and writes
// Y (+ bias), for the CTA at its last segment, whose ring is then idle: the partials of the other
// CTAs gf .. gl are copied into the ring by the bulk-copy engine, as many rows at a time as fit
// (one round trip per chunk instead of one per row), and this CTA's own values come from its
// TMEM accumulator (t_row).  Run by the 128 epilogue threads; returns false when a copy did not
// land in time.
__device__ __forceinline__ bool staged_fixup(const LinearArgs &a, const CUtensorMap *tmap_y, SmemCtl *ctl,
                                             uint8_t *ring, uint32_t ring_bytes, uint8_t *out_stage, int32_t &gi,
                                             int32_t tile, int32_t gf, int32_t gl, int32_t self, bool gf_second,
                                             int32_t rank, uint32_t t_row, int32_t et, int32_t m_local, int32_t o,
                                             bool o_ok, float bias_o, int32_t row0, int32_t rows_c,
                                             volatile int32_t *abort_flag) {
    const int32_t np = gl - gf;  // partials read from global memory
    const uint32_t row_bytes = BM * 4u;
    int32_t cr = static_cast<int32_t>(ring_bytes / (static_cast<uint32_t>(np) * row_bytes)) & ~(kGroupRows - 1);
    cr = min(cr, a.n_tile);
    const int32_t nch = (rows_c + cr - 1) / cr;
    cr = (((rows_c + nch - 1) / nch) + kGroupRows - 1) & ~(kGroupRows - 1);
    const float *staged = reinterpret_cast<const float *>(ring);
    for (int32_t c = 0; c < nch; ++c) {
        const int32_t r0 = c * cr, rc = min(cr, rows_c - r0);
        if (et == 0) {
            fence_proxy_async();  // earlier accesses of the ring before the new copies
            ctl->fix_chunks = c + 1;  // at most one staged sum per launch: phase c
            mbar_arrive_expect_tx(&ctl->fix, static_cast<uint32_t>(np * rc) * row_bytes);
            int32_t pi = 0;
            for (int32_t gg = gf; gg <= gl; ++gg) {
                if (gg == self) continue;
                const int32_t slot = (gg == gf && gf_second) ? 1 : 0;
                const uint8_t *src = reinterpret_cast<const uint8_t *>(part_slot(a, gg, slot, rank) +
                                                                       static_cast<size_t>(r0) * BM);
                uint8_t *dst = ring + static_cast<size_t>(pi) * cr * row_bytes;
                const uint32_t bytes = static_cast<uint32_t>(rc) * row_bytes;
                for (uint32_t off = 0; off < bytes; off += 32768u)
                    bulk_load(dst + off, src + off, min(32768u, bytes - off), &ctl->fix);
                ++pi;
            }
        }
        if (!mbar_wait(&ctl->fix, static_cast<uint32_t>(c) & 1u, abort_flag)) {
            *abort_flag = 1;
            latch(a.status, kDevTimeout);
        }
        named_barrier_sync(1, 128);
        if (*abort_flag) return false;
        for (int32_t n0 = r0; n0 < r0 + rc; n0 += kGroupRows) {
            uint32_t r[kGroupRows];
            __syncwarp();
            tmem_ld_32(t_row + static_cast<uint32_t>(n0), r);
            tmem_wait_ld();
            // a group at a time: every load of the group, then every add, then every store
            const float *src0 = staged + static_cast<size_t>(n0 - r0) * BM + m_local;
            float sum[kGroupRows];
            int32_t pi = 0;
            for (int32_t gg = gf; gg <= gl; ++gg) {
                float v[kGroupRows];
                if (gg == self) {
#pragma unroll
                    for (int j = 0; j < kGroupRows; ++j) v[j] = __uint_as_float(r[j]);
                } else {
                    const float *src = src0 + static_cast<size_t>(pi) * cr * BM;  // rows of the chunk
#pragma unroll
                    for (int j = 0; j < kGroupRows; ++j) v[j] = src[static_cast<size_t>(j) * BM];
                    ++pi;
                }
                if (gg == gf) {
#pragma unroll
                    for (int j = 0; j < kGroupRows; ++j) sum[j] = v[j];
                } else {
#pragma unroll
                    for (int j = 0; j < kGroupRows; ++j) sum[j] += v[j];
                }
            }
            if (a.y_tma) {
#pragma unroll
                for (int j = 0; j < kGroupRows; ++j) sum[j] += bias_o;
                group_store(a, tmap_y, out_stage, gi, et, m_local, sum, true, nullptr, tile, n0, row0, rows_c);
            } else if (o_ok) {
#pragma unroll
                for (int j = 0; j < kGroupRows; ++j)
                    if (n0 + j < r0 + rc) store_y(a, row0 + n0 + j, o, sum[j] + bias_o);
            }
        }
        named_barrier_sync(1, 128);  // every thread is done with the chunk
    }
    return true;
}

// kPair: CTA pairs on tcgen05 .cta_group::2 (launched in clusters of 2; a.pair == 1).
template <int kPair>
__global__ void __launch_bounds__(kThreads, 1)
    linear_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                          const __grid_constant__ CUtensorMap tmap_x,
                          const __grid_constant__ CUtensorMap tmap_y, const LinearArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int32_t stages = a.stages;
    // with pairs each CTA holds half of the activation rows of a stage
    const uint32_t b_bytes = static_cast<uint32_t>(a.n_tile >> kPair) * 128u;
    uint8_t *a_tiles = base;
    uint8_t *b_tiles = base + static_cast<size_t>(stages) * kABytes;
    uint8_t *out_stage = b_tiles + static_cast<size_t>(stages) * b_bytes;  // bulk-store staging
    SmemCtl *ctl = reinterpret_cast<SmemCtl *>(out_stage + a.out_stage_bytes);
    const uint32_t ring_bytes = static_cast<uint32_t>(stages) * (kABytes + b_bytes);
    volatile int32_t *abort_flag = &ctl->abort;

    const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // workers: CTAs, or CTA pairs (the pair's even CTA issues the MMAs for both); the k-block
    // stream runs over the workers' units: tiles, or pairs of adjacent tiles
    const int32_t G = gridDim.x >> kPair, g = blockIdx.x >> kPair;
    const int32_t rank = kPair ? static_cast<int32_t>(blockIdx.x & 1u) : 0;
    const int64_t nkb = a.num_kb;
    const int32_t nch = a.num_chunks;
    const int64_t total = static_cast<int64_t>(a.num_wtiles) * nch * nkb;
    int64_t kb_begin = div_nonneg(total * g, G), kb_end = div_nonneg(total * (g + 1), G);

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->acc_full[i], 1);
            mbar_init(&ctl->acc_empty[i], kPair ? 8 : 4);  // pairs: both CTAs' epilogue warps
        }
        mbar_init(&ctl->fix, 1);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        ctl->is_last = 0;
        ctl->fix_chunks = 0;
        fence_barrier_init();
        prefetch_tensormap(&tmap_w);
        prefetch_tensormap(&tmap_x);
    }
    if (warp == 1) {
        if (kPair) {
            tmem_alloc_pair(&ctl->tmem_base, static_cast<uint32_t>(a.tmem_cols));
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&ctl->tmem_base, static_cast<uint32_t>(a.tmem_cols));
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (kPair) cluster_sync();  // both CTAs' barriers are initialised before either signals the other
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    uint32_t issued = 0, issued_parity = 0;  // producer bookkeeping, for unwinding

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t pol_w = policy_evict_first();  // weights: streamed once
            const uint64_t pol_x = policy_evict_last();   // activation rows: read by every CTA
            // A stage holds one k-block: this CTA's weight tile and its activation rows (all of
            // them, or with pairs this CTA's half).  With pairs both CTAs' loads count on the even
            // CTA's barrier, which expects the bytes of both.
            auto expect = [&](int s) {
                if (!kPair)
                    mbar_arrive_expect_tx(&ctl->full[s], kABytes + b_bytes);
                else if (rank == 0)
                    mbar_arrive_expect_tx(&ctl->full[s], 2u * (kABytes + b_bytes));
            };
            auto load_w = [&](int s, int32_t kx, int32_t unit) {
                uint8_t *dst = a_tiles + static_cast<size_t>(s) * kABytes;
                if (kPair)
                    tma_load_2d_pair(dst, &tmap_w, peer_addr(&ctl->full[s], 0), kx, (2 * unit + rank) * BM, pol_w);
                else
                    tma_load_2d(dst, &tmap_w, &ctl->full[s], kx, unit * BM, pol_w);
            };
            auto load_x = [&](int s, int32_t kx, int32_t chunk) {
                uint8_t *dst = b_tiles + static_cast<size_t>(s) * b_bytes;
                const int32_t y = chunk * a.n_tile;
                if (kPair)
                    tma_load_2d_pair(dst, &tmap_x, peer_addr(&ctl->full[s], 0), kx, y + rank * (a.n_tile >> 1), pol_x);
                else
                    tma_load_2d(dst, &tmap_x, &ctl->full[s], kx, y, pol_x);
            };
            // The weights do not depend on the previous kernel: fill the whole ring with weight
            // tiles first, then wait for the previous kernel and add the activation slices.
            const int64_t n_pre = min(static_cast<int64_t>(stages), kb_end - kb_begin);
            // units are weight-major: unit u covers weight unit u / nch and row chunk u % nch
            for (int64_t i = 0; i < n_pre; ++i) {
                const int64_t kb = kb_begin + i;
                const int32_t unit = static_cast<int32_t>(div_nonneg(kb, nkb));
                const int32_t kx = static_cast<int32_t>(kb - static_cast<int64_t>(unit) * nkb) * BK;
                expect(static_cast<int>(i));
                load_w(static_cast<int>(i), kx, nch == 1 ? unit : unit / nch);
                issued |= 1u << i;
            }
            pdl_wait();
            for (int64_t i = 0; i < n_pre; ++i) {
                const int64_t kb = kb_begin + i;
                const int32_t unit = static_cast<int32_t>(div_nonneg(kb, nkb));
                const int32_t kx = static_cast<int32_t>(kb - static_cast<int64_t>(unit) * nkb) * BK;
                load_x(static_cast<int>(i), kx, nch == 1 ? 0 : unit - (unit / nch) * nch);
            }
            uint32_t stage = static_cast<uint32_t>(n_pre % stages);
            uint32_t phase = (n_pre == stages) ? 1u : 0u;
            for (int64_t kb = kb_begin + n_pre; kb < kb_end; ++kb) {
                const int32_t unit = static_cast<int32_t>(div_nonneg(kb, nkb));
                const int32_t kx = static_cast<int32_t>(kb - static_cast<int64_t>(unit) * nkb) * BK;
                if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    latch(a.status, kDevTimeout);
                    break;
                }
                const int32_t wu = nch == 1 ? unit : unit / nch;
                expect(static_cast<int>(stage));
                load_w(static_cast<int>(stage), kx, wu);
                load_x(static_cast<int>(stage), kx, unit - wu * nch);
                issued |= 1u << stage;
                issued_parity = phase ? (issued_parity | (1u << stage))
                                      : (issued_parity & ~(1u << stage));
                if (++stage == static_cast<uint32_t>(stages)) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (single thread; with pairs, the even CTA's) ----------------
            const uint32_t idesc = idesc_bf16_f32(kPair ? 2 * BM : BM, static_cast<uint32_t>(a.n_tile));
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t kb = kb_begin; kb < kb_end && ok;) {
                const int64_t tile = div_nonneg(kb, nkb);
                const int64_t k1 = min(kb_end, (tile + 1) * nkb);
                if (!mbar_wait(&ctl->acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * static_cast<uint32_t>(a.n_tile);
                for (int64_t k = kb; k < k1; ++k) {
                    if (!mbar_wait(&ctl->full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(a_tiles + static_cast<size_t>(stage) * kABytes);
                    const uint32_t b0 = smem_u32(b_tiles + static_cast<size_t>(stage) * b_bytes);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        if (kPair)
                            mma_bf16_ss_pair(d_tmem, sw128_kmajor_desc(a0 + kk * 32),
                                             sw128_kmajor_desc(b0 + kk * 32), idesc,
                                             (k > kb || kk > 0) ? 1u : 0u);
                        else
                            mma_bf16_ss(d_tmem, sw128_kmajor_desc(a0 + kk * 32),
                                        sw128_kmajor_desc(b0 + kk * 32), idesc,
                                        (k > kb || kk > 0) ? 1u : 0u);
                    }
                    if (kPair)
                        mma_commit_pair_mc(&ctl->empty[stage], 3);  // the stage is free in both CTAs
                    else
                        mma_commit(&ctl->empty[stage]);
                    if (++stage == static_cast<uint32_t>(stages)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (kPair)
                    mma_commit_pair_mc(&ctl->acc_full[acc], 3);  // each CTA drains its own 128 rows
                else
                    mma_commit(&ctl->acc_full[acc]);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
                kb = k1;
            }
            if (!ok) {
                *abort_flag = 1;
                latch(a.status, kDevTimeout);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2..5, TMEM lane quarter = warp % 4 ----------------
        pdl_wait();  // partials, tickets and outputs may still be in use by the previous kernel
        const int32_t q = warp & 3;
        const int32_t m_local = q * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        bool first = true;
        int32_t gi = 0;  // 32-row groups sent by bulk stores
        for (int64_t kb = kb_begin; kb < kb_end;) {
            const int32_t unit = static_cast<int32_t>(div_nonneg(kb, nkb));
            const int32_t wu = nch == 1 ? unit : unit / nch, chunk = unit - wu * nch;
            const int32_t tile = kPair ? 2 * wu + rank : wu;       // this CTA's 128 weight rows
            const int32_t ticket = kPair ? 2 * unit + rank : unit;  // its (weight tile, row chunk)
            const int32_t row0 = chunk * a.n_tile, rows_c = min(a.n_tile, a.rows - row0);
            const int64_t t0 = static_cast<int64_t>(unit) * nkb;
            const int64_t k1 = min(kb_end, t0 + nkb);
            const bool full = (kb == t0) && (k1 == t0 + nkb);
            const bool got = mbar_wait(&ctl->acc_full[acc], acc_phase, abort_flag);
            if (!got) {
                *abort_flag = 1;
                latch(a.status, kDevTimeout);
            }
            dcheck(tile < a.num_tiles, a.status);  // a phantom tile would overrun the tickets
            const int32_t o = tile * BM + m_local;
            const bool o_ok = o < a.M;
            const float bias_o = (a.bias != nullptr && o_ok) ? __bfloat162float(a.bias[o]) : 0.0f;
            // A tile cut between CTAs gf .. gl and summed in this launch.  With owner_fix, the CTA
            // at its last segment that finds every other CTA's ticket in (usually: the head of a
            // tile whose tail the next CTA computed first) owns the sum and takes its own values
            // straight from TMEM; the other CTAs leave partials and tickets.
            const bool split = !full && !a.defer;
            int32_t gf = g, gl = g;
            bool owner = false;
            if (split) {
                gf = cta_of(t0, total, G);
                gl = cta_of(t0 + nkb - 1, total, G);
                if (a.owner_fix) {
                    const bool fits = static_cast<uint32_t>(gl - gf) * kGroupRows * BM * 4u <= ring_bytes;
                    if (threadIdx.x == 64)  // acquire: the other CTAs' partials, for the copies
                        ctl->is_last = (got && !*abort_flag && fits && k1 == kb_end &&
                                        ld_acquire_gpu(&a.counters[ticket]) == gl - gf) ? 1 : 0;
                    named_barrier_sync(1, 128);
                    owner = ctl->is_last != 0;
                }
            }
            // CTAs gf < g <= gl start inside the tile, so it is their first segment (slot 0); CTA
            // gf wrote slot 1 unless its range starts with this tile.
            const bool gf_second = div_nonneg(total * gf, G) < t0;
            __syncwarp();
            if (got && owner) {
                tc_fence_after();
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       acc * static_cast<uint32_t>(a.n_tile);
                staged_fixup(a, &tmap_y, ctl, base, ring_bytes, out_stage, gi, tile, gf, gl, g, gf_second, rank,
                             t_row, threadIdx.x - 64, m_local, o, o_ok, bias_o, row0, rows_c, abort_flag);
            } else if (got) {
                tc_fence_after();
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       acc * static_cast<uint32_t>(a.n_tile);
                float *part = part_slot(a, g, first ? 0 : 1, rank);
                if (a.y_tma) {  // a whole tile into Y, or this CTA's partial, in 32-row groups
                    for (int32_t n0 = 0; n0 < rows_c; n0 += kGroupRows) {
                        uint32_t r[kGroupRows];
                        __syncwarp();
                        tmem_ld_32(t_row + static_cast<uint32_t>(n0), r);
                        tmem_wait_ld();
                        float v[kGroupRows];
#pragma unroll
                        for (int j = 0; j < kGroupRows; ++j) v[j] = __uint_as_float(r[j]) + (full ? bias_o : 0.0f);
                        group_store(a, &tmap_y, out_stage, gi, threadIdx.x - 64, m_local, v, full, part, tile, n0,
                                    row0, rows_c);
                    }
                } else {
                    for (int32_t n0 = 0; n0 < rows_c; n0 += 16) {
                        uint32_t r[16];
                        __syncwarp();
                        tmem_ld_16(t_row + static_cast<uint32_t>(n0), r);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int32_t n = n0 + j;
                            if (n < rows_c) {
                                const float v = __uint_as_float(r[j]);
                                if (full) {
                                    if (o_ok) store_y(a, row0 + n, o, v + bias_o);
                                } else {
                                    part[static_cast<size_t>(n) * BM + m_local] = v;
                                }
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && got) {
                if (kPair)
                    mbar_arrive_cluster(peer_addr(&ctl->acc_empty[acc], 0));  // the issuing CTA's
                else
                    mbar_arrive(&ctl->acc_empty[acc]);
            }
            if (split && owner) {
                if (threadIdx.x == 64) a.counters[ticket] = 0;  // ready for the next launch
                named_barrier_sync(1, 128);                  // ctl->is_last is reused
            } else if (split) {
                named_barrier_sync(1, 128);  // this CTA's partials of the tile are written
                if (threadIdx.x == 64) {
                    if (a.y_tma) {  // the partial went out by bulk stores: complete them first
                        bulk_wait_all();
                        fence_proxy_async();
                    }
                    int32_t last = 0;
                    if (!*abort_flag) {
                        // release: the partials written before the barrier; acquire: the other
                        // CTAs' partials, for the reads after the next barrier
                        const int32_t prev = atomic_add_acq_rel_gpu(&a.counters[ticket], 1);
                        last = (prev == gl - gf);
                        if (last) a.counters[ticket] = 0;  // ready for the next launch
                    }
                    ctl->is_last = last;
                }
                named_barrier_sync(1, 128);
                if (ctl->is_last) {
                    // Sum the partials in ascending CTA order.  Thread e of the 128 sums outputs
                    // 4(e % 32) .. +3 of rows e / 32, +4, +8, ...; all loads of a batch of rows x
                    // CTAs are issued before any is used, so the fix-up costs one L2 round trip
                    // per batch instead of one per (row, CTA).
                    const int32_t et = static_cast<int32_t>(threadIdx.x) - 64;
                    const int32_t m4 = (et & 31) * 4, rsub = et >> 5;
                    float b4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int32_t oq = tile * BM + m4 + q;
                        b4[q] = (a.bias != nullptr && oq < a.M) ? __bfloat162float(a.bias[oq]) : 0.0f;
                    }
                    // 4 rows x 6 CTAs a thread and batch: up to 16 rows all in one batch, so a
                    // tile shared by up to 6 CTAs costs one round trip of loads
                    constexpr int kRowsPerBatch = 4, kCtasPerBatch = 6;  // per thread
                    for (int32_t n0 = rsub; n0 < rows_c; n0 += 4 * kRowsPerBatch) {
                        float4 sum[kRowsPerBatch];
                        for (int32_t g0 = gf; g0 <= gl; g0 += kCtasPerBatch) {
                            float4 x[kCtasPerBatch][kRowsPerBatch];
#pragma unroll
                            for (int c = 0; c < kCtasPerBatch; ++c) {
                                const int32_t gg = g0 + c;
                                const int32_t slot = (gg == gf && gf_second) ? 1 : 0;
                                const float *src = (gg <= gl) ? part_slot(a, gg, slot, rank) + m4 : a.partials;
#pragma unroll
                                for (int j = 0; j < kRowsPerBatch; ++j) {
                                    const int32_t n = n0 + 4 * j;
                                    x[c][j] = (gg <= gl && n < rows_c)
                                                  ? __ldcg(reinterpret_cast<const float4 *>(
                                                        src + static_cast<size_t>(n) * BM))
                                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                                }
                            }
#pragma unroll
                            for (int c = 0; c < kCtasPerBatch; ++c)
#pragma unroll
                                for (int j = 0; j < kRowsPerBatch; ++j) {
                                    if (g0 + c > gl) continue;
                                    if (g0 + c == gf) {
                                        sum[j] = x[c][j];
                                    } else {
                                        sum[j].x += x[c][j].x;
                                        sum[j].y += x[c][j].y;
                                        sum[j].z += x[c][j].z;
                                        sum[j].w += x[c][j].w;
                                    }
                                }
                        }
#pragma unroll
                        for (int j = 0; j < kRowsPerBatch; ++j) {
                            const int32_t n = n0 + 4 * j;
                            if (n >= rows_c) continue;
                            const float v[4] = {sum[j].x, sum[j].y, sum[j].z, sum[j].w};
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (tile * BM + m4 + q < a.M) store_y(a, row0 + n, tile * BM + m4 + q, v[q] + b4[q]);
                        }
                    }
                }
                named_barrier_sync(1, 128);
            }
            if (*abort_flag) break;
            first = false;
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
            kb = k1;
        }
        if (threadIdx.x == 64 && a.y_tma) bulk_wait_all();  // before the staging buffers go away
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_flag) {
        // Unwind after a timeout: let every copy and MMA this CTA started land before the CTA
        // exits and its shared and tensor memory are handed to another CTA.
        if (warp == 0 && lane == 0) {
            if (kPair && rank == 1) {
                // this CTA's loads count on the other CTA's barriers, which it cannot wait on:
                // give them a bounded time to land (a load takes microseconds)
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 200000ull) {
                }
            } else {
                for (int s = 0; s < stages; ++s)
                    if ((issued >> s) & 1u) mbar_wait(&ctl->full[s], (issued_parity >> s) & 1u, nullptr);
            }
            if (ctl->fix_chunks > 0)
                mbar_wait(&ctl->fix, static_cast<uint32_t>(ctl->fix_chunks - 1) & 1u, nullptr);
        }
        if (warp == 1 && lane == 0 && rank == 0) {
            if (kPair)
                mma_commit_pair_mc(&ctl->drain, 1);
            else
                mma_commit(&ctl->drain);
            mbar_wait(&ctl->drain, 0, nullptr);
        }
        __syncwarp();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (kPair) {
        // the issuing CTA's MMAs read this CTA's shared memory and write its tensor memory, and
        // this CTA's epilogue arrives on the issuing CTA's barriers: neither leaves before the
        // other is done
        __syncwarp();
        cluster_sync();
    }
    if (warp == 1) {
        __syncwarp();
        if (kPair)
            tmem_dealloc_pair(tmem_base, static_cast<uint32_t>(a.tmem_cols));
        else
            tmem_dealloc(tmem_base, static_cast<uint32_t>(a.tmem_cols));
    }
}

// ---------------------------------------------------------------------------------------------
// Deferred split-K sum for many rows: block (t, y) adds, for rows y*kReduceRows .. +15 of the
// t-th (weight tile, row chunk) when more than one CTA worked on it, the partials of its CTAs in ascending CTA order (the
// same order and the same sums as the in-kernel fix-up) and writes Y (+ bias).  Thread e sums
// outputs 4(e % 32) .. +3 of rows e / 32 and e / 32 + 8; all its loads are issued together.
// ---------------------------------------------------------------------------------------------
constexpr int kReduceRows = 16;

__global__ void __launch_bounds__(256) linear_reduce_kernel(const LinearArgs a, int32_t G) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t unit = static_cast<int32_t>(blockIdx.x) >> a.pair;  // G counts workers (CTAs or pairs)
    const int32_t rank = static_cast<int32_t>(blockIdx.x) & a.pair;
    const int32_t wu = unit / a.num_chunks, chunk = unit - wu * a.num_chunks;
    const int32_t tile = a.pair ? 2 * wu + rank : wu;
    const int32_t row0 = chunk * a.n_tile, rows_c = min(a.n_tile, a.rows - row0);
    const int64_t nkb = a.num_kb;
    const int64_t total = static_cast<int64_t>(a.num_wtiles) * a.num_chunks * nkb;
    const int64_t t0 = static_cast<int64_t>(unit) * nkb;
    const int32_t gf = cta_of(t0, total, G), gl = cta_of(t0 + nkb - 1, total, G);
    if (gf == gl) return;  // one CTA computed the whole tile and wrote it
    const bool gf_second = div_nonneg(total * gf, G) < t0;
    const int32_t m4 = (threadIdx.x & 31) * 4, rsub = threadIdx.x >> 5;
    constexpr int kCtasPerBatch = 8;
    float4 sum[2];
    for (int32_t g0 = gf; g0 <= gl; g0 += kCtasPerBatch) {
        float4 x[kCtasPerBatch][2];
#pragma unroll
        for (int c = 0; c < kCtasPerBatch; ++c) {
            const int32_t gg = g0 + c;
            const int32_t slot = (gg == gf && gf_second) ? 1 : 0;
            const float *src = (gg <= gl) ? part_slot(a, gg, slot, rank) + m4 : a.partials;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int32_t n = blockIdx.y * kReduceRows + rsub + 8 * j;
                x[c][j] = (gg <= gl && n < rows_c)
                              ? __ldcg(reinterpret_cast<const float4 *>(src + static_cast<size_t>(n) * BM))
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
#pragma unroll
        for (int c = 0; c < kCtasPerBatch; ++c)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (g0 + c > gl) continue;
                if (g0 + c == gf) {
                    sum[j] = x[c][j];
                } else {
                    sum[j].x += x[c][j].x;
                    sum[j].y += x[c][j].y;
                    sum[j].z += x[c][j].z;
                    sum[j].w += x[c][j].w;
                }
            }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int32_t n = blockIdx.y * kReduceRows + rsub + 8 * j;
        if (n >= rows_c) continue;
        const float v[4] = {sum[j].x, sum[j].y, sum[j].z, sum[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int32_t o = tile * BM + m4 + q;
            if (o >= a.M) continue;
            const float b = a.bias != nullptr ? __bfloat162float(a.bias[o]) : 0.0f;
            store_y(a, row0 + n, o, v[q] + b);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// fp32: one warp per output feature, lanes stride the reduction, 8 rows per pass.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    linear_f32_kernel(const float *__restrict__ w, int64_t ldw, const float *__restrict__ x,
                      int64_t ldx, const float *__restrict__ bias, float *__restrict__ y,
                      int64_t ldy, int32_t M, int32_t K, int32_t rows) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t o = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int32_t lane = threadIdx.x & 31;
    if (o >= M) return;
    const float *wr = w + static_cast<int64_t>(o) * ldw;
    const float b = bias ? bias[o] : 0.0f;
    for (int32_t r0 = 0; r0 < rows; r0 += 8) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        for (int32_t i = lane; i < K; i += 32) {
            const float wi = wr[i];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (r0 + j < rows) acc[j] = fmaf(wi, x[static_cast<int64_t>(r0 + j) * ldx + i], acc[j]);
        }
        float mine = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float v = acc[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == j) mine = v;
        }
        if (lane < 8 && r0 + lane < rows) y[static_cast<int64_t>(r0 + lane) * ldy + o] = mine + b;
    }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode_bf16_2d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
    if ((row_stride_elems * 2) % 16 != 0) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_elems * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Y [rows][ldo] (fp32 or bf16) for TMA stores of {box_cols columns, box_rows rows}, no swizzle.
bool encode_out_2d(CUtensorMap *map, const void *ptr, int32_t out_bf16, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_elems, uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    const uint64_t es = out_bf16 ? 2 : 4;
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
    if ((row_stride_elems * es) % 16 != 0) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_elems * es};
    if ((box_cols * es) % 16 != 0 || box_cols > 256 || box_rows > 256 || box_rows < 1) return false;
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, out_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
              const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The output map of a plan: {128, 32} boxes for the epilogue's 32-row groups.
bool encode_plan_out(LinearPlan *p, const void *out) {
    return encode_out_2d(&p->tmap_y, out, p->out_bf16, static_cast<uint64_t>(p->M), static_cast<uint64_t>(p->rows),
                         static_cast<uint64_t>(p->ldo), BM, static_cast<uint32_t>(kGroupRows));
}

}  // namespace

bool encode_bf16_rows_map(CUtensorMap *map, const void *ptr, uint64_t cols, uint64_t rows, uint64_t ld,
                          uint32_t box_cols, uint32_t box_rows) {
    return encode_bf16_2d(map, ptr, cols, rows, ld, box_cols, box_rows);
}

bool encode_kv_cache_map(CUtensorMap *map, const void *cache, int32_t B, int32_t P, int32_t Hk, int32_t D) {
    EncodeTiledFn fn = encoder();
    if (!fn || B < 1 || P < 1 || Hk < 1 || (D != 64 && D != 128)) return false;
    if (reinterpret_cast<uintptr_t>(cache) % 16 != 0) return false;
    // [B][P][Hk][D] bf16 as dims (D, Hk, P, B); one box is 64 head dims of one kv head for 64 keys
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hk), static_cast<cuuint64_t>(P),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hk) * D * 2,
                             static_cast<cuuint64_t>(P) * Hk * D * 2};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(cache), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int32_t linear_n_tile(int32_t rows) { return ((rows + 15) / 16) * 16; }

size_t linear_partials_bytes(int32_t grid, int32_t n_tile) {
    return static_cast<size_t>(grid) * 2 * n_tile * BM * sizeof(float);
}

size_t linear_counters_bytes(int32_t M, int32_t rows) {
    const int64_t chunks = (static_cast<int64_t>(rows < 1 ? 1 : rows) + kLinearMaxRows - 1) / kLinearMaxRows;
    return static_cast<size_t>((M + BM - 1) / BM) * static_cast<size_t>(chunks) * sizeof(int32_t);
}

bool plan_linear_bf16(LinearPlan *p, const void *w, int64_t ldw, int32_t M, int32_t K, const void *x,
                      int64_t ldx, int32_t rows, const void *bias, void *out, int64_t ldo,
                      int32_t out_bf16, float *partials, int32_t *counters, int32_t *status,
                      int32_t num_sms) {
    if (M < 1 || K < 1 || rows < 1 || rows > kLinearMaxLaunchRows || num_sms < 1) return false;
    if (ldw < K || ldx < K || ldo < M) return false;
    p->M = M;
    p->K = K;
    p->rows = rows;
    // more rows than one MMA's N: chunks of kLinearMaxRows rows, each a unit of the split with
    // every weight tile
    p->num_chunks = (rows + kLinearMaxRows - 1) / kLinearMaxRows;
    p->n_tile = linear_n_tile(rows < kLinearMaxRows ? rows : kLinearMaxRows);
    p->num_kb = (K + BK - 1) / BK;
    p->num_tiles = (M + BM - 1) / BM;
    const int64_t total = static_cast<int64_t>(p->num_kb) * p->num_tiles * p->num_chunks;
    p->grid = static_cast<int32_t>(total < num_sms ? total : num_sms);
    // CTA pairs (.cta_group::2) for stream-K above 16 rows when the tiles pair up: the split runs
    // over pairs of adjacent tiles and the grid is twice the pairs
    p->pair = 0;
    p->num_wtiles = p->num_tiles;
    if (rows > kLinearMaxFixupRows && p->num_tiles % 2 == 0) {
        const int32_t pairs = linear_pair_workers(num_sms);
        if (pairs > 0) {
            p->pair = 1;
            p->num_wtiles = p->num_tiles / 2;
            const int64_t total_w = static_cast<int64_t>(p->num_kb) * p->num_wtiles * p->num_chunks;
            p->grid = 2 * static_cast<int32_t>(total_w < pairs ? total_w : pairs);
        }
    }
    const size_t stage_bytes = kABytes + static_cast<size_t>(p->n_tile >> p->pair) * 128;
    // above 16 rows (stream-K), outputs and partials leave in 32-row groups by bulk stores
    const bool want_y_tma = rows > kLinearMaxFixupRows;
    p->out_stage_bytes = want_y_tma ? static_cast<int32_t>(kOutStageBytes) : 0;
    size_t stages = (kMaxDynSmem - 1024 - sizeof(SmemCtl) - p->out_stage_bytes) / stage_bytes;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return false;
    p->stages = static_cast<int32_t>(stages);
    p->smem_bytes = 1024 + stages * stage_bytes + p->out_stage_bytes + sizeof(SmemCtl);
    int32_t cols = 32;
    while (cols < 2 * p->n_tile) cols *= 2;
    p->tmem_cols = cols;
    p->bias = bias;
    p->out = out;
    p->ldo = ldo;
    p->out_bf16 = out_bf16;
    // Many rows: one CTA per tile cannot sum the partials fast enough (it reads CTAs x rows x 128
    // floats); a separate launch spreads the sum over tiles x row blocks.
    // Above 16 rows, split tiles are summed inside the launch when every CTA covers at least a
    // whole tile's k-blocks (then a tile is shared by at most two CTAs, and the one that reaches
    // it at the end of its range finds the other's partial in and owns the sum), else by a
    // second launch.
    const int64_t per_cta =  // fewest of any worker
        static_cast<int64_t>(p->num_kb) * p->num_wtiles * p->num_chunks / (p->grid >> p->pair);
    p->owner_fix = (rows > kLinearMaxFixupRows && per_cta >= p->num_kb) ? 1 : 0;
    p->defer = (rows > kLinearMaxFixupRows && !p->owner_fix) ? 1 : 0;
    p->partials = partials;
    p->counters = counters;
    p->status = status;
    if (!encode_bf16_2d(&p->tmap_w, w, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                        static_cast<uint64_t>(ldw), BK, BM))
        return false;
    p->y_tma = (want_y_tma && encode_plan_out(p, out)) ? 1 : 0;
    if (!encode_bf16_2d(&p->tmap_x, x, static_cast<uint64_t>(K), static_cast<uint64_t>(rows),
                        static_cast<uint64_t>(ldx), BK, static_cast<uint32_t>(p->n_tile >> p->pair)))
        return false;
    return true;
}

// CTA pairs that can be resident at once (clusters of 2 with the largest shared-memory request),
// at most half the SMs; 0 disables pairs (also when EAGLE_LINEAR_PAIR=0 is set in the
// environment, to compare the two ways).  Checked once per device.
int32_t linear_pair_workers(int32_t num_sms) {
    static std::mutex mu;
    static int cached[64] = {};  // 0 unknown, else max active pair clusters + 1
    static const bool disabled = [] {
        const char *e = std::getenv("EAGLE_LINEAR_PAIR");
        return e != nullptr && e[0] == '0';
    }();
    if (disabled) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (prepare_kernels() != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kMaxDynSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, linear_bf16_tc_kernel<1>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cached[dev] = n + 1;
    }
    const int32_t n = cached[dev] - 1;
    return n < num_sms / 2 ? n : num_sms / 2;
}

cudaError_t prepare_kernels() {
    cudaError_t e = cudaFuncSetAttribute(linear_bf16_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMaxDynSmem));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(linear_bf16_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kMaxDynSmem));
}

void linear_retarget_out(LinearPlan *p, void *out) {
    p->out = out;
    if (p->y_tma) p->y_tma = encode_plan_out(p, out) ? 1 : 0;
}

cudaError_t launch_linear_bf16(const LinearPlan &p, cudaStream_t st) {
    LinearArgs a;
    a.M = p.M;
    a.K = p.K;
    a.rows = p.rows;
    a.n_tile = p.n_tile;
    a.num_kb = p.num_kb;
    a.num_tiles = p.num_tiles;
    a.stages = p.stages;
    a.tmem_cols = p.tmem_cols;
    a.bias = reinterpret_cast<const __nv_bfloat16 *>(p.bias);
    a.out = p.out;
    a.ldo = p.ldo;
    a.out_bf16 = p.out_bf16;
    a.defer = p.defer;
    a.owner_fix = p.owner_fix;
    a.pair = p.pair;
    a.num_wtiles = p.num_wtiles;
    a.num_chunks = p.num_chunks;
    a.slots = 2 * p.grid;
    a.y_tma = p.y_tma;
    a.out_stage_bytes = p.out_stage_bytes;
    a.partials = p.partials;
    a.counters = p.counters;
    a.status = p.status;
    cudaError_t e;
    if (p.pair)
        e = launch_pdl_cluster(linear_bf16_tc_kernel<1>, dim3(p.grid), dim3(kThreads), 2u, p.smem_bytes, st,
                               p.tmap_w, p.tmap_x, p.tmap_y, a);
    else
        e = launch_pdl(linear_bf16_tc_kernel<0>, dim3(p.grid), dim3(kThreads), p.smem_bytes, st, p.tmap_w,
                       p.tmap_x, p.tmap_y, a);
    if (e != cudaSuccess || !p.defer) return e;
    return launch_pdl(linear_reduce_kernel, dim3(p.num_tiles * p.num_chunks, (p.n_tile + kReduceRows - 1) / kReduceRows),
                      dim3(256), 0, st, a, p.grid >> p.pair);
}

cudaError_t launch_linear_f32(const float *w, int64_t ldw, const float *x, int64_t ldx,
                              const float *bias, float *y, int64_t ldy, int32_t M, int32_t K,
                              int32_t rows, cudaStream_t st) {
    if (M < 1 || rows < 1) return cudaSuccess;
    const int warps = 8;
    return launch_pdl(linear_f32_kernel, dim3((M + warps - 1) / warps), dim3(warps * 32), 0, st, w, ldw, x,
                      ldx, bias, y, ldy, M, K, rows);
}

}  // namespace eagle
