// decode.cu: paged grouped-query decode attention (pa_decode).
//
// Source: "nano-vLLM Part 4", section 3 (decode: one already-sampled token per sequence,
// attention over its cached history through a block table); "mini-vLLM" (one token per
// sequence attending to that sequence's cached keys and values, grouped-query attention).
//
// Decode reads every cached K/V row once and does ~G multiply-adds per byte, far below the HBM
// ridge, so the kernel is organised to keep HBM streaming, not to reach the tensor cores.
//
// Work: the flattened space of 64-position tiles (128 on the tensor-core path at D = 64) over
// (sequence b, kv head g, tile t), ordered b, then g, then t, is cut into units of contiguous
// tiles: one equal range per persistent CTA (one or two CTAs per SM), so every SM streams about
// the same number of bytes; with one producer warp the last eighth of the tiles is cut into small
// units instead, which CTAs take from a counter as they finish (the dynamic tail), so CTAs on
// slower SMs take fewer of them. A unit covers whole (b, g) pairs plus at most a partial pair at
// each end ("segments"); the merge kernel combines the pieces of pairs split between units.
//
// CTA = 1 or 2 producer warps + 8 consumer warps.
//  * Producer: walks its units; for each tile it looks the rows' physical blocks up in the block
//    table and issues TMA loads of the K and V tile rows (one box per run of `box_rows` rows that
//    share a block) into a ring of shared-memory stages, plus a bulk copy of the G query rows at
//    the start of each segment. full/empty mbarriers hand stages to and from the consumers; the
//    ring (2-6 stages of 32-64 KB) keeps up to ~130 KB per SM in flight across pair boundaries.
//  * Consumers, small groups (G <= 3): warp w owns rows 8w..8w+7 of every 64-row tile. QK: LPP lanes per row, each holding E
//    query elements per head (scaled by scale*log2 e) and multiplying with packed fp32 pairs
//    (two independent passes of 8 rows);
//    the chunk each lane reads depends on the lane so that rows sharing a bank phase hit
//    disjoint banks of the unswizzled tile. Online softmax in base 2 per warp; PV with each lane
//    owning 8 output columns. At a segment's end the 8 warps' (max, sum, O) are combined: a
//    segment covering its whole pair writes the output; a partial segment writes (O/sum, max,
//    sum) to one of its unit's two workspace slots, and decode_merge_kernel combines the pieces.
//  * Consumers, large groups (G >= 4): at ~G multiply-adds per byte the fp32 pipes, not HBM,
//    would set the pace, so the G heads of one KV head go through the warp-level tensor-core
//    path as the M rows of a 16-row fragment (heads G..15 are zero). Per warp and tile:
//    S[16 x 8 rows] = Q K^T with m16n8k16 over D, the online softmax on the score fragment
//    (a quad of lanes holds one head's 8 scores), then O[16 x D] += P V with m16n8k8, P taken
//    straight from the score fragment and the V fragments read transposed by ldmatrix. The K/V
//    tiles land through TMA with the 128-byte swizzle (two 64-column halves when D = 128) so
//    the ldmatrix reads are free of bank conflicts.
//  * Every wait is bounded (PA_DEVERR_TIMEOUT); the producer drains its copies before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>

#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kTN = 64;                  // positions per consumer tile (a stage holds 1 or 2)
constexpr int kConsumers = 8;            // consumer warps
constexpr int kWPos = kTN / kConsumers;  // rows per consumer warp per tile
constexpr int kConsThreads = 32 * kConsumers;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kSmemPerSm = 227 * 1024;
constexpr int kMaxStages = 8;  // the tile metas and barriers of 8 stages fit their 1 KB
constexpr int kLook = 2;                     // a producer's steps prepared ahead of the one it issues
constexpr int kIdRing = 4;                   // each producer's ring of prepared tiles (> kLook)
static_assert(kIdRing > kLook && (kIdRing & (kIdRing - 1)) == 0, "block-id ring");

struct PrepTile {
    int b, g, t, n, nt, unit, flags, pad;  // b < 0: no tile (the CTA's work is done)
};
// tensor-core consumers from this group size on
constexpr int kMmaMinGroup = 4;
template <int G>
constexpr bool use_mma() { return G >= kMmaMinGroup; }
// persistent CTAs per SM: two (two TMA streams, 16 consumer warps) when the consumers fit the
// halved register file, else one
__host__ __device__ constexpr int ctas_per_sm(int D, int G) { return G < kMmaMinGroup ? 2 : 1; }
// The D = 64 tensor-core kernels also come with two CTAs per SM (half the stages each, twice the
// producers per SM): faster on large batches, slower on small ones, where the longer pipeline
// start of each CTA is not paid back. Chosen per launch from an upper bound of the stages per SM.
constexpr int kWideMinStagesPerSm = 32;
__host__ __device__ constexpr bool has_wide(int D, int G) { return G >= kMmaMinGroup && D == 64; }
// producer warps (alternate tiles): two keep the light tensor-core consumers fed; with the fp32
// consumers one suffices and a second only takes issue slots from them
__host__ __device__ constexpr int producers_for(int D, int G) { return G < kMmaMinGroup ? 1 : 2; }
__host__ __device__ constexpr int threads_for(int D, int G) { return 32 * (producers_for(D, G) + kConsumers); }

// flags of one tile
constexpr int kFirst = 1;  // first tile of a segment: reset the state, read q
constexpr int kLast = 2;   // last tile of a segment: combine the warps and write
constexpr int kWhole = 4;  // the segment is its pair's whole context: write the output
constexpr int kSlot1 = 8;  // partial segment that is not the unit's first: workspace slot 1
constexpr int kEnd = 16;   // no tile: the CTA's work is done (dynamic tail)

// Dynamic tail (kernels with one producer warp). The launch's tiles [0, F) are cut into one equal
// contiguous unit per CTA, as in the static scheme; the last 1/kTailDiv of them, [F, total), into
// K2 units (at most kTailUnitsPerCta per CTA) of 1/32 of a CTA's share, 2 to 8 tiles, that CTAs
// take from a counter as they finish, so that CTAs on slower SMs take fewer of them. All unit
// bounds are closed-form, so the merge finds the pieces of a pair without a list.
constexpr int kTailDiv = 8;
constexpr int kTailUnitsPerCta = 8;
constexpr int kDynMinTilesPerCta = 16;  // smaller launches keep the static scheme
constexpr int kDynCoarse = 32;          // batches beyond one CTA's threads: offsets per 32 sequences

struct TileMeta {
    int b, g, flags, all_valid;  // all_valid: every one of the 128 rows is a context position
    unsigned long long valid[2];  // bit r of the 128-bit mask: tile row r is a context position
    int newrow, unit;             // row whose K/V are in the spare row (a new token), or -1;
                                  // the unit the tile belongs to
};

// What the merge kernel needs to know about one unit of work (a CTA's static range, or one
// unit of the dynamic tail).
struct SegRecord {
    long long lo, hi;        // the unit's tile range
    long long pair_start;    // global index of the first tile of the unit's first pair
    long long total;         // tiles in the whole launch
    long long F;             // tiles in the static units (total without a dynamic tail)
    int b, g, ntiles;        // that pair and its tile count; b < 0: empty range
    int P, K2;               // static units (= CTAs) and tail units of the launch
    unsigned epoch;          // the launch that wrote the record
};

struct DecodeParams {
    CUtensorMap tmap_k, tmap_v;  // [slots, Hkv, D] views of the pools, box [box_rows, 1, D]
    const void *q;
    const void *k_new, *v_new;  // fused store: the new tokens' rows [B, Hkv, D], or null
    void *k_cache, *v_cache;    // the pools (written by the fused store only)
    const int32_t *block_tables, *context_lens;
    void *out;
    float *part;     // [units][2][G][D + 2]: normalised O, max (log2 units), sum
    SegRecord *rec;  // [units]
    unsigned long long *ctr;  // dynamic tail: [0] epoch tag, [1] tickets handed out (low word)
    int32_t *err;
    int B, Hq, Hkv, max_blocks, num_blocks, box_rows, stages;
    int tail_units;  // units of the dynamic tail the workspace holds (0: static scheme only)
    unsigned epoch;  // distinct for every launch (never 0)
    BlockGeom geom;
    float scale_log2;
};

template <int D, int G, int CPS_ = ctas_per_sm(D, G)>
struct Shape {
    static constexpr int NCH = D / 8;  // 16-byte chunks per row
    static constexpr int CPS = CPS_;
    // QK elements per lane: keeps the query registers (G * E) at 32 with two CTAs per SM,
    // at 64 with one
    static constexpr int E_RAW = CPS == 2 ? (G == 1 ? 32 : G == 2 ? 16 : 8) : (G <= 4 ? 16 : 8);
    static constexpr int E = E_RAW < D / 4 ? E_RAW : D / 4;  // QK elements per lane
    static constexpr int LPP = D / E;                         // lanes per row in QK
    static constexpr int PPP = 32 / LPP;                      // rows per QK pass
    static constexpr int PASSES = kWPos / PPP;
    static constexpr int CPL = E / 8;                         // chunks per lane in QK
    static constexpr int CPV = G >= 6 ? 4 : 8;                // PV output columns per lane
    static constexpr int NPV = CPV / 2;                       // ... as fp32 pairs
    static constexpr int LPR = D / CPV;                       // PV lanes per row
    static constexpr int RPI = 32 / LPR;                      // PV rows per instruction
    static constexpr int PV_IT = kWPos / RPI;
    static constexpr int HPR = 32 / kWPos;                    // softmax heads per round
    static constexpr int ROUNDS = (G + HPR - 1) / HPR;
    static constexpr bool MMA = use_mma<G>();
    // positions per stage: 128 for the tensor-core path at D = 64 (as many bytes per stage, and as
    // much producer work per byte, as at D = 128), else 64; consumers take it 64 rows at a time
    static constexpr int TN = (MMA && D == 64) ? 2 * kTN : kTN;
    static constexpr int SUB = TN / kTN;
    static constexpr int LANE_BOXES = TN / 32;  // TMA boxes per producer lane and stage, at most
    static constexpr int NH = D / 64;  // 64-column halves of a swizzled tile
    // one swizzled tile half: TN rows + the spare row, 128 bytes each. The 128-byte swizzle is a
    // function of the shared-memory address (16-byte chunk c of the 128-byte line at address a
    // sits at c ^ ((a >> 7) & 7)), so halves need only 128-byte alignment and readers take the
    // phase from the address.
    static constexpr int SW_HALF = (TN + 1) * 128;
    // 64 rows + a spare row that takes a new token's K (or V) row in the fused store + decode;
    // tensor-core consumers: NH swizzled halves of 128-byte rows
    static constexpr int TILE_BYTES = MMA ? NH * SW_HALF : (TN + 1) * D * 2;
    static constexpr int Q_BYTES = G * D * 2;
    // stages on 1 KB boundaries for the unswizzled tiles; 128 bytes suffice for the swizzled ones
    static constexpr int STAGE_ALIGN = MMA ? 128 : 1024;
    static constexpr int STAGE_BYTES = (2 * TILE_BYTES + Q_BYTES + STAGE_ALIGN - 1) / STAGE_ALIGN * STAGE_ALIGN;
    static constexpr int RED_BYTES = kConsumers * G * (D + 2) * 4;
    // scores, probabilities and rescale factors of the fp32 consumers
    static constexpr int SCRATCH_BYTES = MMA ? 0 : 2 * kConsumers * G * kWPos * 4 + kConsumers * G * 4;
    static_assert(PASSES >= 1 && PPP * PASSES == kWPos, "QK mapping");
    static_assert(RPI * PV_IT == kWPos, "PV mapping");
    // chunk that lane (row u of a pass, part r) reads at step c. With 4 lanes per row two rows
    // share an 8-lane bank phase: they take opposite 64-byte halves of each 128-byte group.
    static __device__ __forceinline__ int chunk(int c, int r, int u) {
        if (LPP == 4) return 8 * (c >> 1) + 4 * ((c & 1) ^ (u & 1)) + r;
        return c * LPP + r;
    }
};

// the dynamic tail's tile offsets (int32: one per sequence, or one per 32 sequences)
__host__ __device__ constexpr int dyn_seq_bytes(int D, int G) {
    return producers_for(D, G) == 1 ? (threads_for(D, G) + 1 + 1) / 2 * 8 : 0;
}

template <int D, int G, int CPS>
constexpr int fixed_smem() {
    // + metas, barriers, scan scratch (1 KB), the slack that aligns the ring (1 KB) and the
    // producer's ring of prepared tiles
    using S = Shape<D, G, CPS>;
    return S::RED_BYTES + S::SCRATCH_BYTES + 2048 + producers_for(D, G) * kIdRing * (S::TN * 4 + 32) +
           dyn_seq_bytes(D, G);
}

// All 32 lanes wait for the phase, then the warp reconverges; false (for every lane) if the wait
// ran out or the CTA is aborting.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const bool ok = mbar_wait(bar, parity) && !*abort_flag;
    const bool all = __all_sync(kFull, ok);
    __syncwarp();
    return all;
}

// validity of the kWPos rows of consumer warp cw in 64-row sub-tile `sub`, as the low bits of a word
__device__ __forceinline__ unsigned warp_rows_valid(const TileMeta &m, int cw, int sub = 0) {
    const int first = sub * kTN + cw * kWPos;
    const unsigned long long w = m.valid[first >> 6];
    return static_cast<unsigned>(w >> (first & 63)) & ((1u << kWPos) - 1u);
}

// ldmatrix: four 8x8 matrices of 16-bit elements; lane 8j + i gives the address of row i of
// matrix j, and register j of lane l holds (row l / 4, columns 2 (l % 4), +1) of matrix j
// (transposed: rows 2 (l % 4), +1 of column l / 4)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d += A B with A 16 x 16 (row-major fragment; rows 8..15 zero, so only a0 and a2 are passed)
// and B 16 x 8, fp32 accumulation
template <class E>
__device__ __forceinline__ void mma_k16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    if constexpr (E::kIsBf16)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
// d += A B with A 16 x 8 and B 8 x 8
template <class E>
__device__ __forceinline__ void mma_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    if constexpr (E::kIsBf16)
        asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(b0));
    else
        asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(b0));
}

// stages of TN positions over sequence b's context
// The next ticket of this launch from the dynamic tail's counter: 0, 1, 2, ... in the order CTAs
// ask, one atomic add each. The counter is reset once per launch, by whichever CTA asks first: the
// tag word holds the epoch of the launch the counter belongs to (with bit 32 set while a CTA is
// resetting it), so a word another launch left, or one never written, is reset before use and the
// workspace needs no clearing between launches. `ready` (per CTA) remembers that this launch's
// reset has been seen. -1 if the wait for another CTA's reset ran out.
__device__ __forceinline__ long long take_ticket(unsigned long long *tag, unsigned *cnt, unsigned epoch,
                                                 bool &ready) {
    if (!ready) {
        const unsigned long long mine = epoch, resetting = (1ull << 32) | epoch;
        unsigned long long t = *reinterpret_cast<volatile unsigned long long *>(tag);
        const uint64_t t0 = globaltimer_ns();
        for (int it = 0;; ++it) {
            if (t == mine) break;
            if (t != resetting) {
                const unsigned long long prev = atomicCAS(tag, t, resetting);
                if (prev == t) {  // this CTA resets the counter
                    atomicExch(cnt, 0u);
                    __threadfence();
                    atomicExch(tag, mine);
                    break;
                }
                t = prev;
                continue;
            }
            if ((it & 15) == 15 && globaltimer_ns() - t0 > kWaitLimitNs) return -1;
            __nanosleep(64);
            t = *reinterpret_cast<volatile unsigned long long *>(tag);
        }
        __threadfence();
        ready = true;
    }
    return static_cast<long long>(atomicAdd(cnt, 1u));
}

template <int TN>
__device__ __forceinline__ int ntiles_of(const DecodeParams &p, int b, long long cap) {
    const int n = p.context_lens[b];
    if (n <= 0 || n > cap) return 0;
    return (n + TN - 1) / TN;
}

// block-wide sum over all NT threads; `red` holds NT / 32 longs
template <int NT>
__device__ long long block_sum(long long v, long long *red) {
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    long long t = 0;
    for (int i = 0; i < NT / 32; ++i) t += red[i];
    __syncthreads();
    return t;
}

template <int D, int G, class E, int CPS>
__global__ void __launch_bounds__(threads_for(D, G), CPS) decode_kernel(const __grid_constant__ DecodeParams p) {
    using S = Shape<D, G, CPS>;
    constexpr int kProducers = producers_for(D, G), kThreads = threads_for(D, G);
    using T = typename E::T;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // stages start on a 1024-byte boundary (the launch adds 1 KB of slack for this)
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int NS = p.stages;
    unsigned char *ring = smem;
    float *red = reinterpret_cast<float *>(smem + NS * S::STAGE_BYTES);  // [8][G][D+2]
    float *sbuf = red + kConsumers * G * (D + 2);                        // [8][G][16] scores
    float *pbuf = sbuf + kConsumers * G * kWPos;                         // [8][G][16] probs
    float *abuf = pbuf + kConsumers * G * kWPos;                         // [8][G] rescale
    TileMeta *metas = reinterpret_cast<TileMeta *>(reinterpret_cast<unsigned char *>(sbuf) + S::SCRATCH_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(metas + NS);  // full[NS], empty[NS], cons[2]
    long long *scan = reinterpret_cast<long long *>(bars + 2 * NS + 2);  // 16 longs + start
    volatile int *abort_flag = reinterpret_cast<volatile int *>(scan + 20);
    PrepTile *prep = reinterpret_cast<PrepTile *>(scan + 24);  // [producers][kIdRing]
    int *idring = reinterpret_cast<int *>(prep + kProducers * kIdRing);  // [producers][kIdRing][TN]
    int *seqpre = idring + kProducers * kIdRing * S::TN;  // dynamic tail: first tile of each
                                                          // sequence (or of every 32nd)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, cta = blockIdx.x;
    const long long cap = static_cast<long long>(p.max_blocks) * p.geom.block_size;
    // the merge kernel may be launched now: it waits for this grid's completion before it reads
    // anything, so only its launch overlaps this grid (it is also why the wait below comes after
    // the shared-memory setup: that part overlaps the grid before this one)
    asm volatile("griddepcontrol.launch_dependents;");
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + NS),
                   cons0 = smem_addr(bars + 2 * NS);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumers);
        }
        mbar_init(cons0, kConsumers);
        mbar_init(cons0 + 8, kConsumers);
        *abort_flag = 0;
        fence_mbar_init();
    }

    // launched as a programmatic dependent: nothing this grid reads may be touched before the
    // grids it depends on have completed
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // zero rows of a sequence without positions (and flag lengths outside the table)
    auto check_seq = [&](int b, int n) -> int {
        if ((n < 0 || n > cap) && b % P == cta) raise_err(p.err, PA_DEVERR_LENGTH);
        const int nt = (n <= 0 || n > cap) ? 0 : (n + S::TN - 1) / S::TN;
        if (nt == 0 && b % P == cta) {
            uint4 *o = reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + static_cast<size_t>(b) * p.Hq * D);
            for (int i = 0; i < p.Hq * D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
        }
        return nt;
    };
    long long total, lo, hi;
    if (p.B <= kThreads) {
        // ---- one pass: each thread one sequence; a block scan of the tile counts gives the
        // total and the (b, g, t) of tile `lo` ----
        const int nt = tid < p.B ? check_seq(tid, p.context_lens[tid]) : 0;
        long long v = nt;  // inclusive scan of nt across the block
        for (int o = 1; o < 32; o <<= 1) {
            const long long x = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += x;
        }
        if (lane == 31) scan[warp] = v;
        if (tid == 0) scan[16] = -1;
        __syncthreads();
        long long before = 0, all = 0;
        for (int i = 0; i < kThreads / 32; ++i) {
            if (i < warp) before += scan[i];
            all += scan[i];
        }
        total = all * p.Hkv;
        lo = total * cta / P;
        hi = total * (cta + 1) / P;
        const long long excl = (before + v - nt) * p.Hkv;
        if (lo < hi && nt > 0 && excl <= lo && lo < excl + static_cast<long long>(nt) * p.Hkv) {
            scan[16] = tid;
            scan[17] = excl;
        }
        if constexpr (kProducers == 1) {
            if (total < (1ll << 31)) {  // the only case the dynamic tail runs in
                if (tid < p.B) seqpre[tid] = static_cast<int>(excl);
                if (tid == 0) seqpre[p.B] = static_cast<int>(total);
            }
        }
        __syncthreads();
    } else {
        // ---- pass 1: tiles per sequence, the total ----
        long long mine = 0;
        for (int b = tid; b < p.B; b += kThreads) mine += check_seq(b, p.context_lens[b]);
        total = block_sum<kThreads>(mine, scan) * p.Hkv;
        lo = total * cta / P;
        hi = total * (cta + 1) / P;
        // the dynamic tail needs the first tile of every 32nd sequence: pass 2 then runs to the end
        const bool coarse = kProducers == 1 && p.tail_units > 0 && p.B <= kDynCoarse * kThreads &&
                            total < (1ll << 31) && total >= static_cast<long long>(kDynMinTilesPerCta) * P;

        // ---- pass 2: the (b, g, t) of tile `lo` ----
        if (tid == 0) scan[16] = -1;
        __syncthreads();
        if (lo < hi || coarse) {
            long long running = 0;  // tiles of sequences before this chunk, times Hkv
            for (int base = 0; base < p.B; base += kThreads) {
                const int b = base + tid;
                const int nt = b < p.B ? ntiles_of<S::TN>(p, b, cap) : 0;
                long long v = nt;  // inclusive scan of nt across the block
                for (int o = 1; o < 32; o <<= 1) {
                    const long long x = __shfl_up_sync(kFull, v, o);
                    if (lane >= o) v += x;
                }
                if (lane == 31) scan[warp] = v;
                __syncthreads();
                long long before = 0, chunk_total = 0;
                for (int i = 0; i < kThreads / 32; ++i) {
                    if (i < warp) before += scan[i];
                    chunk_total += scan[i];
                }
                const long long excl = running + (before + v - nt) * p.Hkv;
                if (lo < hi && nt > 0 && excl <= lo && lo < excl + static_cast<long long>(nt) * p.Hkv) {
                    scan[16] = b;
                    scan[17] = excl;
                }
                if (coarse && b < p.B && b % kDynCoarse == 0) seqpre[b / kDynCoarse] = static_cast<int>(excl);
                running += chunk_total * p.Hkv;
                __syncthreads();
                if (!coarse && running > lo) break;  // uniform: every thread sees the same `running`
            }
            if (coarse && tid == 0) seqpre[(p.B + kDynCoarse - 1) / kDynCoarse] = static_cast<int>(total);
        }
        __syncthreads();
    }
    const int b0 = static_cast<int>(scan[16]);
    const long long seq_start = scan[17];  // global index of tile (b0, 0, 0)

    // the dynamic tail runs for large enough launches of at most 32 CTAs' threads of sequences
    // (their tile offsets, per sequence or per 32 sequences, live in shared memory) when the
    // workspace holds its units; the choice is the same in every CTA
    bool dyn = false;
    long long F = total;
    int K2 = 0;
    if (kProducers == 1 && p.tail_units > 0 && p.B <= kDynCoarse * kThreads && total < (1ll << 31) &&
        total >= static_cast<long long>(kDynMinTilesPerCta) * P) {
        F = total - total / kTailDiv;
        const long long per_cta = total / P;  // tiles of a CTA's share
        const long long chunk = per_cta / 32 < 2 ? 2 : (per_cta / 32 > 8 ? 8 : per_cta / 32);
        const long long k2 = (total - F + chunk - 1) / chunk;
        K2 = static_cast<int>(k2 < p.tail_units ? k2 : p.tail_units);
        dyn = K2 > 0;
        if (!dyn) F = total;
    }
    const bool exact_seq = p.B <= kThreads;  // seqpre holds every sequence's first tile
    auto make_rec = [&](long long ulo, long long uhi) {
        SegRecord r{};
        r.lo = ulo;
        r.hi = uhi;
        r.total = total;
        r.F = F;
        r.P = P;
        r.K2 = K2;
        r.epoch = p.epoch;
        r.b = -1;
        return r;
    };
    if (!dyn) {
        if (tid == 0) {
            SegRecord r = make_rec(lo, hi);
            if (lo < hi && b0 >= 0) {
                const int nt = ntiles_of<S::TN>(p, b0, cap);
                const long long off = lo - seq_start;
                r.b = b0;
                r.g = static_cast<int>(off / nt);
                r.ntiles = nt;
                r.pair_start = seq_start + static_cast<long long>(r.g) * nt;
            }
            p.rec[cta] = r;
        }
        if (lo >= hi || b0 < 0) return;
    }
    const long long count = hi - lo;  // static scheme: the CTA's tiles

    if (warp < kProducers) {
        // ======================= producers =======================
        // producer pw issues tiles i = pw, pw + kProducers, ... (stage i % NS: with NS a multiple
        // of kProducers every stage has one producer)
        const int pw = warp;
        if (lane == 0) {
            prefetch_tmap(&p.tmap_k);
            prefetch_tmap(&p.tmap_v);
        }
        constexpr int TN = S::TN;
        const int R = p.box_rows, nbox = TN / R;
        const uint32_t box_bytes = static_cast<uint32_t>(R) * D * 2;
        const unsigned long long box_rows_mask = R == 64 ? ~0ull : ((1ull << R) - 1ull);
        // The unit being walked: `u_count` tiles; the walker (b, g, t) is the next tile to
        // prepare, `u_pos` its index in the unit. The unit's first segment is its tiles
        // [0, first_len); it began inside its pair if first_mid. With the dynamic tail (one
        // producer) the CTA's stream of tiles runs through unit after unit; `stream_total` counts
        // the tiles of the units taken so far.
        long long unit = cta, u_count = 0, u_pos = pw, first_len = 0, stream_total = 0;
        bool first_mid = false, done = false, took_static = false, ticket_ready = false;
        int b = 0, nt = 1, n = 0, g = 0, t = 0;
        auto seed = [&](int sb, long long sstart, long long X, long long cnt) {
            b = sb;
            nt = ntiles_of<S::TN>(p, b, cap);
            n = p.context_lens[b];
            const long long off = X - sstart;
            g = static_cast<int>(off / nt);
            t = static_cast<int>(off % nt);
            u_count = cnt;
            first_len = min(cnt, static_cast<long long>(nt - t));
            first_mid = t > 0;
        };
        auto advance = [&]() {
            if (++t == nt) {
                t = 0;
                if (++g == p.Hkv) {
                    g = 0;
                    do {
                        ++b;
                    } while (b < p.B && (nt = ntiles_of<S::TN>(p, b, cap)) == 0);
                    if (b < p.B) n = p.context_lens[b];
                }
            }
        };
        // dynamic tail: bounds of unit v (static units first, then the tail's)
        auto unit_lo = [&](long long v) -> long long {
            return v <= P ? F * v / P : F + (total - F) * (v - P) / K2;
        };
        // dynamic tail: the sequence holding tile X and its first tile (offsets are
        // non-decreasing). Per-sequence offsets: a binary search. Offsets per 32 sequences: a
        // binary search for the group, then one warp-wide read of the group's lengths. Warp-uniform.
        auto find_seq = [&](long long X, long long &soff) -> int {
            if (exact_seq) {
                int l = 0, h = p.B;  // seqpre[l] <= X < seqpre[h]
                while (h - l > 1) {
                    const int mid = (l + h) >> 1;
                    if (seqpre[mid] <= X) l = mid;
                    else h = mid;
                }
                soff = seqpre[l];
                return l;
            }
            int l = 0, h = (p.B + kDynCoarse - 1) / kDynCoarse;
            while (h - l > 1) {
                const int mid = (l + h) >> 1;
                if (seqpre[mid] <= X) l = mid;
                else h = mid;
            }
            const int bb = l * kDynCoarse + lane;
            const int ntl = bb < p.B ? ntiles_of<S::TN>(p, bb, cap) : 0;
            int incl = ntl;  // inclusive scan over the group
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            const long long ex = seqpre[l] + static_cast<long long>(incl - ntl) * p.Hkv;
            // the group holds tile X, so its first sequence with tiles starts at or before X
            const unsigned m = __ballot_sync(kFull, ntl > 0 && ex <= X);
            const int ln = 31 - __clz(m);
            soff = __shfl_sync(kFull, ex, ln);
            return l * kDynCoarse + ln;
        };
        // dynamic tail: move the walker to the first tile of the next unit that holds tiles, or
        // set `done`: the CTA's static unit first, then tickets. Records every unit taken (empty
        // ones included). Warp-uniform.
        auto next_unit = [&]() {
            for (;;) {
                long long v;
                if (!took_static) {
                    took_static = true;
                    v = cta;
                } else {
                    long long tk = 0;
                    if (lane == 0)
                        tk = take_ticket(p.ctr, reinterpret_cast<unsigned *>(p.ctr + 1), p.epoch, ticket_ready);
                    tk = __shfl_sync(kFull, tk, 0);
                    if (tk < 0 && lane == 0) {
                        raise_err(p.err, PA_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    if (tk < 0 || tk >= K2) {
                        done = true;
                        return;
                    }
                    v = P + tk;
                }
                const long long vlo = unit_lo(v), vhi = unit_lo(v + 1);
                SegRecord r = make_rec(vlo, vhi);
                if (vlo < vhi) {
                    long long soff;
                    const int sb = find_seq(vlo, soff);
                    seed(sb, soff, vlo, vhi - vlo);
                    unit = v;
                    r.b = b;
                    r.g = g;
                    r.ntiles = nt;
                    r.pair_start = soff + static_cast<long long>(g) * nt;
                }
                if (lane == 0) p.rec[v] = r;
                if (vlo < vhi) return;
            }
        };
        if (!dyn) {
            seed(b0, seq_start, lo, count);
            for (int k = 0; k < pw && k < count; ++k) advance();
        }
        PrepTile *myprep = prep + pw * kIdRing;
        int *myids = idring + pw * kIdRing * TN;
        // Each producer prepares its tiles kLook of its own steps ahead of the one it issues:
        // preparing records the tile's coordinates and flags and queues cp.async copies of its
        // block ids (lane l: boxes l and l + 32) into a ring in shared memory, so the block-table
        // reads are in flight while earlier tiles are issued. Every step commits one cp.async
        // group per lane. With the dynamic tail a step past the CTA's last tile records "no tile".
        auto prepare = [&](long long j) {
            const int sl = static_cast<int>(j % kIdRing);
            // past the unit: on to the next, at the same distance beyond its start
            while (dyn && !done && u_pos >= u_count) {
                const long long carry = u_pos - u_count;
                next_unit();
                if (done) break;
                stream_total += u_count;
                u_pos = carry;
                if (carry < u_count)
                    for (long long c = 0; c < carry; ++c) advance();
            }
            if (done) {
                if (lane == 0) myprep[sl].b = -1;
                cp_async_commit();
                return;
            }
            const bool first = u_pos == 0 || t == 0;
            const bool last = u_pos == u_count - 1 || t == nt - 1;
            const bool in_first = u_pos < first_len;
            int flags = (first ? kFirst : 0) | (last ? kLast : 0);
            // the segment covers its whole pair: it ends the pair and began at the pair's start
            if (last && t == nt - 1 && !(in_first && first_mid)) flags |= kWhole;
            if (!in_first) flags |= kSlot1;
            if (lane == 0) myprep[sl] = PrepTile{b, g, t, n, nt, static_cast<int>(unit), flags, 0};
            const int pos0 = t * TN;
            const int nvalid = min(TN, n - pos0);
#pragma unroll
            for (int k2 = 0; k2 < S::LANE_BOXES; ++k2) {
                const int k = lane + 32 * k2;
                if (k < nbox && k * R < nvalid)
                    cp_async4(smem_addr(myids + sl * TN + k),
                              p.block_tables + static_cast<size_t>(b) * p.max_blocks + p.geom.block_of(pos0 + k * R));
            }
            cp_async_commit();
            u_pos += kProducers;
#pragma unroll
            for (int k = 0; k < kProducers; ++k) advance();
        };
        const long long my_count =
            dyn ? (1ll << 62) : (count > pw ? (count - pw + kProducers - 1) / kProducers : 0);
        for (int j = 0; j < kLook; ++j) {
            if (j < my_count) prepare(j);
            else cp_async_commit();
        }
        long long last_i = -1;  // the last tile this producer issued
        long long j = 0;
        bool aborted = false;
        for (; j < my_count; ++j) {
            const long long i = pw + static_cast<long long>(kProducers) * j;
            if (__shfl_sync(kFull, lane == 0 ? *abort_flag : 0, 0)) {  // warp-uniform
                aborted = true;
                break;
            }
            if (j + kLook < my_count) prepare(j + kLook);
            else cp_async_commit();
            const int stage = static_cast<int>(i % NS);
            const uint32_t phase = static_cast<uint32_t>((i / NS) & 1);
            // everything up to the copies is worked out before the stage is free
            cp_async_wait<kLook>();  // this lane's block ids of tile i have landed
            __syncwarp();
            const int sl = static_cast<int>(j % kIdRing);
            const PrepTile pm = myprep[sl];
            if (pm.b < 0) break;  // dynamic tail: no tiles left
            const int pb_ = pm.b, pg = pm.g, pt = pm.t, pn = pm.n, pnt = pm.nt;
            const int pos0 = pt * TN;
            const int nvalid = min(TN, pn - pos0);
            int slots[S::LANE_BOXES];
            unsigned good[S::LANE_BOXES], badm[S::LANE_BOXES];
#pragma unroll
            for (int k2 = 0; k2 < S::LANE_BOXES; ++k2) {
                const int k = lane + 32 * k2;
                slots[k2] = -1;
                bool bad = false;
                if (k < nbox && k * R < nvalid) {
                    const int id = myids[sl * TN + k];
                    if (id >= 0 && id < p.num_blocks)
                        slots[k2] = id * p.geom.block_size + p.geom.offset_of(pos0 + k * R);
                    else
                        bad = true;
                }
                good[k2] = __ballot_sync(kFull, slots[k2] >= 0);
                badm[k2] = __ballot_sync(kFull, bad);
            }
            // rows holding context positions: [0, nvalid), minus the boxes of ids outside the pool
            // (128-bit mask; a box never straddles its 64-bit word: R divides 64)
            unsigned long long vm0 = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
            unsigned long long vm1 = 0ull;
            if constexpr (TN == 128) vm1 = nvalid >= 128 ? ~0ull : nvalid > 64 ? ((1ull << (nvalid - 64)) - 1ull) : 0ull;
            unsigned nbad = 0, ngood = 0;
#pragma unroll
            for (int k2 = 0; k2 < S::LANE_BOXES; ++k2) {
                nbad += __popc(badm[k2]);
                ngood += __popc(good[k2]);
            }
            if (nbad) {  // rare: flagged, and those rows are masked
                if (lane == 0) raise_err(p.err, PA_DEVERR_TABLE);
#pragma unroll
                for (int k2 = 0; k2 < S::LANE_BOXES; ++k2)
                    for (unsigned m = badm[k2]; m; m &= m - 1) {
                        const int r0 = (32 * k2 + __ffs(m) - 1) * R;
                        if (TN == 64 || r0 < 64) vm0 &= ~(box_rows_mask << r0);
                        else vm1 &= ~(box_rows_mask << (r0 - 64));
                    }
            }
            uint32_t bytes = ngood * 2u * box_bytes;
            const int flags = pm.flags;
            const bool first = (flags & kFirst) != 0;
            if (first) bytes += S::Q_BYTES;
            // fused store: the pair's last tile holds the new token (position pn - 1); its rows
            // come from k_new / v_new into the spare rows, not from the pool
            const bool new_tok = p.k_new != nullptr && pt == pnt - 1;
            if (new_tok) bytes += 2 * D * 2;

            // every lane waits and the warp reconverges before going on (a lane-0-only wait
            // leaves the warp split for the rest of the iteration)
            const bool ok = warp_wait(empty0 + 8 * stage, phase ^ 1, abort_flag);
            if (!ok) {
                if (lane == 0) {
                    raise_err(p.err, PA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                aborted = true;
                break;
            }
            unsigned char *st = ring + static_cast<size_t>(stage) * S::STAGE_BYTES;
            if (lane == 0) {
                TileMeta m;
                m.b = pb_;
                m.g = pg;
                m.flags = flags;
                m.all_valid = vm0 == ~0ull && (TN == 64 || vm1 == ~0ull);
                m.valid[0] = vm0;
                m.valid[1] = vm1;
                m.newrow = new_tok ? (pn - 1) - pos0 : -1;
                m.unit = pm.unit;
                metas[stage] = m;
                mbar_arrive_expect_tx(full0 + 8 * stage, bytes);
            }
            __syncwarp();
            const uint32_t kdst = smem_addr(st), vdst = kdst + S::TILE_BYTES;
#pragma unroll
            for (int k2 = 0; k2 < S::LANE_BOXES; ++k2) {
                const int k = lane + 32 * k2;
                if (slots[k2] >= 0) {
                    if constexpr (S::MMA) {
                        // one box per 64-column half, 128-byte rows, swizzled
#pragma unroll
                        for (int hf = 0; hf < S::NH; ++hf) {
                            const uint32_t o = hf * S::SW_HALF + k * R * 128;
                            tma_load_3d(kdst + o, &p.tmap_k, 64 * hf, pg, slots[k2], full0 + 8 * stage);
                            tma_load_3d(vdst + o, &p.tmap_v, 64 * hf, pg, slots[k2], full0 + 8 * stage);
                        }
                    } else {
                        tma_load_3d(kdst + k * box_bytes, &p.tmap_k, 0, pg, slots[k2], full0 + 8 * stage);
                        tma_load_3d(vdst + k * box_bytes, &p.tmap_v, 0, pg, slots[k2], full0 + 8 * stage);
                    }
                }
            }
            if (first && lane == 0) {
                const T *qsrc = static_cast<const T *>(p.q) + (static_cast<size_t>(pb_) * p.Hq + pg * G) * D;
                bulk_load(kdst + 2 * S::TILE_BYTES, qsrc, S::Q_BYTES, full0 + 8 * stage);
            }
            if (new_tok) {
                const size_t row_off = (static_cast<size_t>(pb_) * p.Hkv + pg) * D;
                if (lane == 0) {
                    if constexpr (S::MMA) {
                        // row TN of each half, copied in as it is (readers take phase 0 there)
#pragma unroll
                        for (int hf = 0; hf < S::NH; ++hf) {
                            const uint32_t o = hf * S::SW_HALF + TN * 128;
                            bulk_load(kdst + o, static_cast<const T *>(p.k_new) + row_off + 64 * hf, 128,
                                      full0 + 8 * stage);
                            bulk_load(vdst + o, static_cast<const T *>(p.v_new) + row_off + 64 * hf, 128,
                                      full0 + 8 * stage);
                        }
                    } else {
                        bulk_load(kdst + TN * D * 2, static_cast<const T *>(p.k_new) + row_off, D * 2,
                                  full0 + 8 * stage);
                        bulk_load(vdst + TN * D * 2, static_cast<const T *>(p.v_new) + row_off, D * 2,
                                  full0 + 8 * stage);
                    }
                }
                // ... and into the pool, at the slot of position pn - 1 (no copy in this launch
                // reads that slot's row: the tile takes it from the spare row)
                const int id = myids[sl * TN + (pn - 1 - pos0) / R];  // its box's block
                constexpr int kChunks = D * 2 / 16;  // 16-byte chunks per row
                if (id >= 0 && id < p.num_blocks && lane < 2 * kChunks) {
                    const long long slot = static_cast<long long>(id) * p.geom.block_size + p.geom.offset_of(pn - 1);
                    const bool is_v = lane >= kChunks;
                    const int c = lane % kChunks;
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                                           static_cast<const T *>(is_v ? p.v_new : p.k_new) + row_off) + c;
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(is_v ? p.v_cache : p.k_cache) +
                                                           (static_cast<size_t>(slot) * p.Hkv + pg) * D) + c;
                    *dst = *src;
                }
            }
            last_i = i;
        }
        // no copy (TMA or block id) may still be in flight when the CTA exits: wait for the
        // tiles this producer issued in the last NS tiles
        cp_async_wait<0>();
        if (lane == 0 && last_i >= 0) {
            for (long long i = last_i; i >= 0 && i > last_i - NS; i -= kProducers) {
                if (!mbar_wait(full0 + 8 * static_cast<int>(i % NS), static_cast<uint32_t>((i / NS) & 1))) {
                    raise_err(p.err, PA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
        }
        __syncwarp();
        const long long i_end = pw + static_cast<long long>(kProducers) * j;
        if (dyn && !aborted && i_end == stream_total) {
            // tell the consumers there is nothing more: the stage after the last tile (this
            // producer's, as its predecessor in that stage was), with no bytes and the end flag,
            // after the drain above, whose waits would not see phases this one completes
            const long long i = i_end;
            const int stage = static_cast<int>(i % NS);
            const uint32_t phase = static_cast<uint32_t>((i / NS) & 1);
            if (warp_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) {
                if (lane == 0) {
                    metas[stage].flags = kEnd;
                    mbar_arrive(full0 + 8 * stage);
                }
            } else if (lane == 0) {
                raise_err(p.err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        return;
    }

    // ========================= consumers =========================
    const int cw = warp - kProducers;  // 0..7
    int seg = 0;   // segments finished (parity of the consumer barriers)
    // Once every consumer warp has put its (max, sum, O) of a finished segment into `red`:
    // combine the 8 warps and write the output (a whole pair) or the CTA's partial. False if
    // a wait ran out.
    auto combine = [&](int mflags, int mb, int mg, int munit) -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(cons0);
        bool ok = warp_wait(cons0, seg & 1, abort_flag);
        if (!ok) {
            if (lane == 0) {
                raise_err(p.err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            return false;
        }
        const int ct = cw * 32 + lane;
        const size_t bh = static_cast<size_t>(mb) * p.Hq + static_cast<size_t>(mg) * G;
        float *part = p.part + (static_cast<size_t>(munit) * 2 + ((mflags & kSlot1) ? 1 : 0)) * G * (D + 2);
        for (int idx = ct; idx < G * D; idx += kConsThreads) {
            const int h = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, red[(w * G + h) * (D + 2) + D]);
            const float mu = M == -INFINITY ? 0.f : M;
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float *rw = red + (w * G + h) * (D + 2);
                const float sc = fast_exp2(rw[D] - mu);
                L = fmaf(rw[D + 1], sc, L);
                O = fmaf(rw[d], sc, O);
            }
            const float o = L > 0.f ? O / L : 0.f;
            if (mflags & kWhole) {
                static_cast<T *>(p.out)[(bh + h) * D + d] = T(o);
            } else {
                part[h * (D + 2) + d] = o;
                if (d == 0) {
                    part[h * (D + 2) + D] = M;
                    part[h * (D + 2) + D + 1] = L;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(cons0 + 8);
        ok = warp_wait(cons0 + 8, seg & 1, abort_flag);
        if (!ok) {
            if (lane == 0) {
                raise_err(p.err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            return false;
        }
        ++seg;
        return true;
    };
    if constexpr (S::MMA) {
        // ---- tensor-core consumers ----
        constexpr int KS = D / 16;  // QK k-steps; also PV m-blocks (16 output columns each)
        const int gq = lane >> 2, tq = lane & 3;  // fragment row (head) and column pair
        const int lr = lane & 7, lm = lane >> 3;  // ldmatrix: row of the warp's 8, matrix index
        uint32_t qa[KS][2];  // Q as the A fragment (rows 8..15 are zero and not held)
        float acc[KS][4];    // O^T: lane holds columns 16i + gq, +8 of heads 2tq, 2tq + 1
        float m_run = -INFINITY, l_part = 0.f;
        int stage = 0;
        uint32_t phase = 0;
        for (long long i = 0; dyn || i < count; ++i) {
            const bool ok = warp_wait(full0 + 8 * stage, phase, abort_flag);
            if (!ok) {
                if (lane == 0) {
                    raise_err(p.err, PA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                return;
            }
            const TileMeta &m = metas[stage];
            const int mflags = m.flags, mb = m.b, mg = m.g, mall = m.all_valid, mnew = m.newrow, munit = m.unit;
            if (mflags & kEnd) break;  // dynamic tail: the CTA's work is done
            const unsigned char *st = ring + static_cast<size_t>(stage) * S::STAGE_BYTES;
            const uint32_t kb = smem_addr(st), vb = kb + S::TILE_BYTES;

            if (mflags & kFirst) {
                const uint32_t *qs = reinterpret_cast<const uint32_t *>(st + 2 * S::TILE_BYTES);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qa[ks][0] = gq < G ? qs[gq * (D / 2) + 8 * ks + tq] : 0u;
                    qa[ks][1] = gq < G ? qs[gq * (D / 2) + 8 * ks + 4 + tq] : 0u;
                }
#pragma unroll
                for (int j = 0; j < KS; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
                m_run = -INFINITY;
                l_part = 0.f;
            }
#pragma unroll
            for (int sub = 0; sub < S::SUB; ++sub) {  // 64-row sub-tiles of the stage
                const unsigned vrows = warp_rows_valid(m, cw, sub);
                // the row this lane addresses in ldmatrix: row lr of the warp's 8, or the spare row
                // that holds the new token (copied in unswizzled: phase 0)
                const int row0 = sub * kTN + cw * kWPos + lr;
                const int row = row0 == mnew ? S::TN : row0;
                const uint32_t rbase = static_cast<uint32_t>(row) * 128u;
                const bool spare = row == S::TN;
                // 128-byte swizzle phase of this row in each half of K and V: (address >> 7) & 7
                auto swz = [&](uint32_t a) -> uint32_t { return spare ? 0u : ((a >> 7) & 7u); };

                // ---- S = Q K^T: this lane gets head gq at the warp's rows 2tq, 2tq + 1 ----
                float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {  // chunks 4q .. 4q + 3 (columns 32q .. 32q + 31)
                    uint32_t r4[4];
                    const uint32_t a = kb + (q >> 1) * S::SW_HALF + rbase;
                    ldsm_x4(a + (((4u * (q & 1) + lm) ^ swz(a)) << 4), r4);
                    mma_k16<E>(s0, qa[2 * q][0], qa[2 * q][1], r4[0], r4[1]);
                    mma_k16<E>(s1, qa[2 * q + 1][0], qa[2 * q + 1][1], r4[2], r4[3]);
                }
                const bool v0 = (vrows >> (2 * tq)) & 1u, v1 = (vrows >> (2 * tq + 1)) & 1u;
                const float x0 = v0 ? (s0[0] + s1[0]) * p.scale_log2 : -INFINITY;
                const float x1 = v1 ? (s0[1] + s1[1]) * p.scale_log2 : -INFINITY;

                // ---- online softmax (base 2) over the warp's 8 rows: a quad holds one head ----
                float mt = fmaxf(x0, x1);
                mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
                const float m_new = fmaxf(m_run, mt);
                const float mu = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = fast_exp2(m_run - mu);
                const float p0 = fast_exp2(x0 - mu), p1 = fast_exp2(x1 - mu);
                m_run = m_new;
                l_part = fmaf(l_part, alpha, p0 + p1);
                // P^T as the B fragment of O^T += V^T P^T: the score fragment's layout as it stands
                const uint32_t pb = E::pack2(p0, p1);
                // the rescale factors of this lane's two O^T columns (heads 2tq, 2tq + 1)
                const float al0 = __shfl_sync(kFull, alpha, 8 * tq), al1 = __shfl_sync(kFull, alpha, 8 * tq + 4);

                // ---- O^T = alpha O^T + V^T P^T, V^T read transposed by ldmatrix; rows outside the
                // context are zeroed in the V fragment (their stage bytes may hold anything, and
                // 0 * NaN is NaN) ----
                const uint32_t keep = mall ? 0xffffffffu : ((v0 ? 0x0000ffffu : 0u) | (v1 ? 0xffff0000u : 0u));
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t r4[4];
                    const uint32_t a = vb + (q >> 1) * S::SW_HALF + rbase;
                    ldsm_x4_t(a + (((4u * (q & 1) + lm) ^ swz(a)) << 4), r4);
#pragma unroll
                    for (int hb = 0; hb < 2; ++hb) {
                        float(&a)[4] = acc[2 * q + hb];
                        a[0] *= al0;
                        a[1] *= al1;
                        a[2] *= al0;
                        a[3] *= al1;
                        mma_k8<E>(a, r4[2 * hb] & keep, r4[2 * hb + 1] & keep, pb);
                    }
                }
            }  // sub-tiles
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * stage);
            if (++stage == NS) {
                stage = 0;
                phase ^= 1;
            }
            if (!(mflags & kLast)) continue;

            // ---- end of a segment: this warp's (max, sum, O) of each head into `red` ----
            float l = l_part;
            l += __shfl_xor_sync(kFull, l, 1);
            l += __shfl_xor_sync(kFull, l, 2);
            if (gq < G && tq == 0) {
                float *rh = red + (cw * G + gq) * (D + 2);
                rh[D] = m_run;
                rh[D + 1] = l;
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int h = 2 * tq + hh;
                if (h < G) {
                    float *rh = red + (cw * G + h) * (D + 2);
#pragma unroll
                    for (int j = 0; j < KS; ++j) {
                        rh[16 * j + gq] = acc[j][hh];
                        rh[16 * j + gq + 8] = acc[j][2 + hh];
                    }
                }
            }
            if (!combine(mflags, mb, mg, munit)) return;
        }
    } else {
        const int r = lane % S::LPP;
        const int rg = lane / S::LPR, cc = lane % S::LPR;
        // softmax: lane handles row spos of heads shead + HPR * k (HPR = 32 / rows per warp)
        const int spos = lane % kWPos, shead = lane / kWPos;
        float *sb = sbuf + cw * G * kWPos;
        float *pb = pbuf + cw * G * kWPos;
        float *ab = abuf + cw * G;

        uint64_t q2[G][S::CPL][4];
        uint64_t acc[G][S::NPV];
        float m_run[S::ROUNDS], l_part[S::ROUNDS];
        int stage = 0;
        uint32_t phase = 0;

        for (long long i = 0; dyn || i < count; ++i) {
            bool ok = warp_wait(full0 + 8 * stage, phase, abort_flag);
            if (!ok) {
                if (lane == 0) {
                    raise_err(p.err, PA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                return;
            }
            const TileMeta &m = metas[stage];
            const int mflags = m.flags, mb = m.b, mg = m.g, mall = m.all_valid, mnew = m.newrow, munit = m.unit;
            if (mflags & kEnd) break;  // dynamic tail: the CTA's work is done
            const unsigned char *st = ring + static_cast<size_t>(stage) * S::STAGE_BYTES;
            const uint32_t kb = smem_addr(st), vb = kb + S::TILE_BYTES;
            // this warp's rows as a validity mask (bit rl: row rl of the warp)
            const unsigned vrows = warp_rows_valid(m, cw);

            if (mflags & kFirst) {
                const T *qs = reinterpret_cast<const T *>(st + 2 * S::TILE_BYTES);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int c = 0; c < S::CPL; ++c) {
                        const int j = S::chunk(c, r, (lane / S::LPP));
                        const uint4 u = *reinterpret_cast<const uint4 *>(qs + h * D + j * 8);
                        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = E::unpack2(w[e]);
                            q2[h][c][e] = f2_pack(f.x * p.scale_log2, f.y * p.scale_log2);
                        }
                    }
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < S::NPV; ++e) acc[h][e] = 0;
#pragma unroll
                for (int k = 0; k < S::ROUNDS; ++k) {
                    m_run[k] = -INFINITY;
                    l_part[k] = 0.f;
                }
            }

            // ---- scores of this warp's 16 rows ----
#pragma unroll
            for (int pass = 0; pass < S::PASSES; ++pass) {
                const int u = lane / S::LPP;
                const int rl = pass * S::PPP + u;  // row within the warp's 16
                const int row = cw * kWPos + rl;
                uint64_t d2[G][S::CPL];
#pragma unroll
                for (int c = 0; c < S::CPL; ++c) {
                    const uint4 kv = lds128(kb + (row == mnew ? S::TN : row) * D * 2 + S::chunk(c, r, u) * 16);
                    const uint64_t k0 = unpack_pair<E>(kv.x), k1 = unpack_pair<E>(kv.y);
                    const uint64_t k2 = unpack_pair<E>(kv.z), k3 = unpack_pair<E>(kv.w);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        uint64_t a = f2_mul(q2[h][c][0], k0);
                        a = f2_fma(q2[h][c][1], k1, a);
                        a = f2_fma(q2[h][c][2], k2, a);
                        d2[h][c] = f2_fma(q2[h][c][3], k3, a);
                    }
                }
                float dot[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    // pairwise tree over the chunks keeps the dependency chain short
                    uint64_t t2 = d2[h][0];
#pragma unroll
                    for (int c = 1; c < S::CPL; ++c) t2 = f2_add(t2, d2[h][c]);
                    dot[h] = f2_lo(t2) + f2_hi(t2);
                }
#pragma unroll
                for (int o = S::LPP / 2; o >= 1; o >>= 1)
#pragma unroll
                    for (int h = 0; h < G; ++h) dot[h] += __shfl_xor_sync(kFull, dot[h], o);
                if (r == 0) {
                    const bool valid = (vrows >> rl) & 1u;
#pragma unroll
                    for (int h = 0; h < G; ++h) sb[h * kWPos + rl] = valid ? dot[h] : -INFINITY;
                }
            }
            __syncwarp();

            // ---- online softmax over the 16 rows ----
#pragma unroll
            for (int k = 0; k < S::ROUNDS; ++k) {
                const int h = shead + S::HPR * k;
                const bool act = h < G;
                const float s = act ? sb[h * kWPos + spos] : -INFINITY;
                float mt = s;
#pragma unroll
                for (int o = kWPos / 2; o >= 1; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o));
                const float m_new = fmaxf(m_run[k], mt);
                const float mu = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = fast_exp2(m_run[k] - mu);
                m_run[k] = m_new;
                const float pr = fast_exp2(s - mu);
                l_part[k] = fmaf(l_part[k], alpha, pr);
                if (act) {
                    pb[h * kWPos + spos] = pr;
                    if (spos == 0) ab[h] = alpha;
                }
            }
            __syncwarp();

            // ---- O = alpha O + P V ----
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float al = ab[h];
                const uint64_t a2 = f2_pack(al, al);
#pragma unroll
                for (int e = 0; e < S::NPV; ++e) acc[h][e] = f2_mul(acc[h][e], a2);
            }
            auto pv_row = [&](int rl) {
                const int row0 = cw * kWPos + rl;
                const int row = row0 == mnew ? S::TN : row0;
                uint64_t v[S::NPV];
                if constexpr (S::CPV == 8) {
                    const uint4 vv = lds128(vb + row * D * 2 + cc * 16);
                    v[0] = unpack_pair<E>(vv.x);
                    v[1] = unpack_pair<E>(vv.y);
                    v[2] = unpack_pair<E>(vv.z);
                    v[3] = unpack_pair<E>(vv.w);
                } else {
                    const uint2 vv = lds64(vb + row * D * 2 + cc * 8);
                    v[0] = unpack_pair<E>(vv.x);
                    v[1] = unpack_pair<E>(vv.y);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float pr = pb[h * kWPos + rl];
                    const uint64_t p2 = f2_pack(pr, pr);
#pragma unroll
                    for (int e = 0; e < S::NPV; ++e) acc[h][e] = f2_fma(p2, v[e], acc[h][e]);
                }
            };
            if (mall) {
#pragma unroll
                for (int it = 0; it < S::PV_IT; ++it) pv_row(it * S::RPI + rg);
            } else {
                // rows outside the context are skipped: their stage bytes may hold anything
#pragma unroll
                for (int it = 0; it < S::PV_IT; ++it) {
                    const int rl = it * S::RPI + rg;
                    if ((vrows >> rl) & 1u) pv_row(rl);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * stage);
            if (++stage == NS) {
                stage = 0;
                phase ^= 1;
            }

            if (!(mflags & kLast)) continue;

            // ---- end of a segment: combine the 8 warps ----
            float *ro = red + cw * G * (D + 2);
#pragma unroll
            for (int k = 0; k < S::ROUNDS; ++k) {
                float l = l_part[k];
#pragma unroll
                for (int o = kWPos / 2; o >= 1; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
                const int h = shead + S::HPR * k;
                if (h < G && spos == 0) {
                    ro[h * (D + 2) + D] = m_run[k];
                    ro[h * (D + 2) + D + 1] = l;
                }
            }
#pragma unroll
            for (int o = S::LPR; o < 32; o <<= 1)
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < S::NPV; ++e) {
                        const float lo_ = f2_lo(acc[h][e]) + __shfl_xor_sync(kFull, f2_lo(acc[h][e]), o);
                        const float hi_ = f2_hi(acc[h][e]) + __shfl_xor_sync(kFull, f2_hi(acc[h][e]), o);
                        acc[h][e] = f2_pack(lo_, hi_);
                    }
            if (rg == 0)
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float *dst = ro + h * (D + 2) + cc * S::CPV;
#pragma unroll
                    for (int e = 0; e < S::NPV; ++e) {
                        dst[2 * e] = f2_lo(acc[h][e]);
                        dst[2 * e + 1] = f2_hi(acc[h][e]);
                    }
                }
            if (!combine(mflags, mb, mg, munit)) return;
        }
    }
}

// One CTA per unit of decode work (a decode CTA's static range, or a unit of the dynamic tail): if
// the unit's first pair began in an earlier unit and ends in this one, combine the pair's partial
// segments into the output. Unit bounds are closed-form (from the record: the launch's tile count,
// the static part F, P static units and K2 tail units), so the list of contributing units (and
// which of each one's two partial slots holds the pair) follows from this unit's own record with
// no further reads. After that record, every global read the result depends on (each segment's
// max, sum and partial row) is issued together: two memory round trips for up to kMergeChunk
// segments. Records this launch did not write are ignored.
constexpr int kMergeMaxCtas = 512;  // decode CTAs per launch (2 per SM at most)
constexpr int kMergeThreads = 256;
constexpr int kMergeBatch = 512;    // contributing units listed at a time

template <int D, int G, class E>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const __grid_constant__ DecodeParams p) {
    using T = typename E::T;
    constexpr int kOut = (G * D + kMergeThreads - 1) / kMergeThreads;  // outputs per thread
    constexpr int kMergeChunk = kOut <= 2 ? 8 : 4;                     // segments loaded at once
    __shared__ int seg_part[kMergeBatch];  // contributing segments: partial slot index, in unit order
    __shared__ int nseg_s;
    const int c = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    // what follows in the stream may launch now (it waits for this grid before reading)
    asm volatile("griddepcontrol.launch_dependents;");
    // launched ahead of time (programmatic dependent launch): wait until the decode grid has
    // completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the decode grid is done with the tail's counter: clear its tag, so that the next launch on
    // this workspace resets the counter even when it carries the same epoch (a replayed graph)
    if (c == 0 && tid == 0) p.ctr[0] = 0ull;
    const SegRecord rc = p.rec[c];
    // unit 0's record is written by every launch: a record this launch did not write (another
    // launch's, or one from an earlier replay of the same graph) disagrees with it or lies past
    // the launch's units
    const SegRecord r0 = p.rec[0];
    if (rc.epoch != p.epoch || r0.epoch != p.epoch || rc.total != r0.total || rc.F != r0.F ||
        rc.P != r0.P || rc.K2 != r0.K2 || c >= r0.P + r0.K2)
        return;
    if (rc.b < 0 || rc.b >= p.B || rc.g < 0 || rc.g >= p.Hkv || rc.P < 1 || rc.K2 < 0 || rc.total <= 0)
        return;
    if (rc.pair_start >= rc.lo || rc.pair_start + rc.ntiles > rc.hi) return;
    const long long x = rc.pair_start, total = rc.total, F = rc.F;
    const int P = rc.P, K2 = rc.K2;
    // unit v holds tiles [lo(v), lo(v + 1))
    auto lo_of = [&](long long v) -> long long {
        return v <= P ? F * v / P : F + (total - F) * (v - P) / K2;
    };
    // first unit whose range holds the pair's first tile: max{v : lo(v) <= pair_start}, from the
    // linear piece (static units below F, tail units above) that holds it
    long long c0l;
    if (x < F) c0l = ((x + 1) * P + F - 1) / F - 1;
    else c0l = P + ((x - F + 1) * K2 + (total - F) - 1) / (total - F) - 1;
    const int c0 = static_cast<int>(c0l < 0 ? 0 : (c0l > c ? c : c0l));
    int hh[kOut], dd[kOut];
    float M[kOut], L[kOut], O[kOut];
#pragma unroll
    for (int j = 0; j < kOut; ++j) {
        const int idx = tid + j * kMergeThreads;
        hh[j] = idx < G * D ? idx / D : -1;
        dd[j] = idx % D;
        M[j] = -INFINITY;
        L[j] = 0.f;
        O[j] = 0.f;
    }
    for (int vbase = c0; vbase <= c; vbase += kMergeBatch) {
        const int vend = min(c, vbase + kMergeBatch - 1);
        if (tid < 32) {  // the units in [vbase, vend] that hold tiles (a unit can be empty)
            int n = 0;
            for (int base = vbase; base <= vend; base += 32) {
                const int v = base + lane;
                const long long lo = v <= vend ? lo_of(v) : 0;
                const bool has = v <= vend && lo < lo_of(v + 1);
                // the pair is the last segment of unit c0 when that unit began in an earlier pair
                // (slot 1), and the first segment of every later unit (slot 0)
                const int slot = (v == c0 && lo < x) ? 1 : 0;
                const unsigned m = __ballot_sync(kFull, has);
                if (has) seg_part[n + __popc(m & ((1u << lane) - 1u))] = 2 * v + slot;
                n += __popc(m);
            }
            if (lane == 0) nseg_s = n;
        }
        __syncthreads();
        const int nseg = nseg_s;
        for (int k0 = 0; k0 < nseg; k0 += kMergeChunk) {
            float mv[kOut][kMergeChunk], lv[kOut][kMergeChunk], ov[kOut][kMergeChunk];
#pragma unroll
            for (int k = 0; k < kMergeChunk; ++k) {
                const bool in = k0 + k < nseg;
                const float *seg = in ? p.part + static_cast<size_t>(seg_part[k0 + k]) * G * (D + 2) : nullptr;
#pragma unroll
                for (int j = 0; j < kOut; ++j) {
                    if (in && hh[j] >= 0) {
                        const float *row = seg + hh[j] * (D + 2);
                        mv[j][k] = row[D];
                        lv[j][k] = row[D + 1];
                        ov[j][k] = row[dd[j]];
                    } else {
                        mv[j][k] = -INFINITY;
                        lv[j][k] = 0.f;
                        ov[j][k] = 0.f;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kOut; ++j) {
                // the running (max, sum, weighted row) of the segments so far, rescaled to the new max
                float cm = M[j];
#pragma unroll
                for (int k = 0; k < kMergeChunk; ++k) cm = fmaxf(cm, mv[j][k]);
                const float mu = cm == -INFINITY ? 0.f : cm;
                const float s = M[j] == -INFINITY ? 0.f : fast_exp2(M[j] - mu);
                float l = L[j] * s, o = O[j] * s;
#pragma unroll
                for (int k = 0; k < kMergeChunk; ++k) {
                    const float w = mv[j][k] == -INFINITY ? 0.f : lv[j][k] * fast_exp2(mv[j][k] - mu);
                    l += w;
                    o = fmaf(w, ov[j][k], o);
                }
                M[j] = cm;
                L[j] = l;
                O[j] = o;
            }
        }
        __syncthreads();  // seg_part is rebuilt for the next batch
    }
    const size_t bh = static_cast<size_t>(rc.b) * p.Hq + static_cast<size_t>(rc.g) * G;
#pragma unroll
    for (int j = 0; j < kOut; ++j)
        if (hh[j] >= 0)
            static_cast<T *>(p.out)[(bh + hh[j]) * D + dd[j]] = T(L[j] > 0.f ? O[j] / L[j] : 0.f);
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// swizzled: boxes of 64 columns with the 128-byte swizzle (tensor-core consumers); else whole
// unswizzled rows
bool encode_pool(CUtensorMap *m, const void *pool, pa_dtype dt, int D, int Hkv, long long slots,
                 int box_rows, bool swizzled) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                          static_cast<cuuint64_t>(slots > 0 ? slots : 1)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hkv) * D * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(swizzled ? 64 : D), 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              // L2 fills no wider than one head's row: a 256-byte fill of a 128-byte row (D = 64)
              // also pulls in the next head's row, which another tile reads much later (measured:
              // 1.44x the KV bytes from DRAM)
              D * 2 >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// encode_pool through a small per-thread cache: a tensor map is a pure function of its
// arguments, so a hit is exact (also after a pool is freed and another one takes its address)
bool encode_pool_cached(CUtensorMap *m, const void *pool, pa_dtype dt, int D, int Hkv, long long slots,
                        int box_rows, bool swizzled) {
    struct Entry {
        const void *pool;
        long long slots;
        int dt, D, Hkv, box_rows, swizzled, valid;
        CUtensorMap map;
    };
    constexpr int kEntries = 8;
    thread_local Entry cache[kEntries] = {};
    thread_local int next = 0;
    for (int i = 0; i < kEntries; ++i) {
        const Entry &e = cache[i];
        if (e.valid && e.pool == pool && e.slots == slots && e.dt == static_cast<int>(dt) && e.D == D &&
            e.Hkv == Hkv && e.box_rows == box_rows && e.swizzled == static_cast<int>(swizzled)) {
            *m = e.map;
            return true;
        }
    }
    if (!encode_pool(m, pool, dt, D, Hkv, slots, box_rows, swizzled)) return false;
    Entry &e = cache[next];
    next = (next + 1) % kEntries;
    e = Entry{pool, slots, static_cast<int>(dt), D, Hkv, box_rows, static_cast<int>(swizzled), 1, *m};
    return true;
}

template <int D, int G, int CPS>
constexpr int stages_for() {
    const int budget = kSmemPerSm / CPS - 1024;
    // A multiple of the producer count, so that each stage belongs to one producer. (A stage that
    // alternated between producers could not be waited on by parity: a producer cannot tell
    // whether the other has armed the stage's previous phase yet, and a barrier two phases behind
    // has the parity of the phase it waits for.)
    constexpr int np = producers_for(D, G);
    const int s = (budget - fixed_smem<D, G, CPS>()) / Shape<D, G, CPS>::STAGE_BYTES / np * np;
    return s < kMaxStages / np * np ? s : kMaxStages / np * np;
}

template <int D, int G, class E, int CPS = ctas_per_sm(D, G)>
cudaError_t launch_typed(DecodeParams &prm, cudaStream_t stream) {
    static_assert(stages_for<D, G, CPS>() >= 2, "the ring needs two stages");
    prm.stages = stages_for<D, G, CPS>();
    const int smem = prm.stages * Shape<D, G, CPS>::STAGE_BYTES + fixed_smem<D, G, CPS>();
    auto kern = decode_kernel<D, G, E, CPS>;
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (configured[dev] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = smem;
    }
    const int P = device_sm_count() * CPS;
    if (P > kMergeMaxCtas) return cudaErrorInvalidConfiguration;
    // both kernels launch as programmatic dependents of what precedes them in the stream: a
    // launch overlaps the tail of the grid before it, and each kernel waits on the grid
    // dependency before it reads anything
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t dcfg{};
    dcfg.gridDim = dim3(P);
    dcfg.blockDim = dim3(threads_for(D, G));
    dcfg.dynamicSmemBytes = smem;
    dcfg.stream = stream;
    dcfg.attrs = attr;
    dcfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&dcfg, kern, prm);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(P + prm.tail_units);  // one merge CTA per unit
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D, G, E>, prm);
}

template <int D, int G, class E>
cudaError_t launch_group(bool wide, DecodeParams &prm, cudaStream_t stream) {
    if constexpr (has_wide(D, G))
        if (wide) return launch_typed<D, G, E, 2>(prm, stream);
    return launch_typed<D, G, E>(prm, stream);
}

template <int D, class E>
cudaError_t dispatch_group(int G, bool wide, DecodeParams &prm, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_group<D, 1, E>(wide, prm, stream);
        case 2: return launch_group<D, 2, E>(wide, prm, stream);
        case 3: return launch_group<D, 3, E>(wide, prm, stream);
        case 4: return launch_group<D, 4, E>(wide, prm, stream);
        case 5: return launch_group<D, 5, E>(wide, prm, stream);
        case 6: return launch_group<D, 6, E>(wide, prm, stream);
        case 7: return launch_group<D, 7, E>(wide, prm, stream);
        case 8: return launch_group<D, 8, E>(wide, prm, stream);
        default: return cudaErrorInvalidValue;
    }
}

// CTAs per SM of a launch: the kernel's own, or two for the D = 64 tensor-core kernels when the
// batch may give each SM at least kWideMinStagesPerSm stages (an upper bound: every sequence at
// the table's full length)
int launch_ctas_per_sm(int B, int Hq, int Hkv, int D, int max_blocks_per_seq, int block_size,
                       bool allow_wide) {
    const int G = Hq / Hkv;
    if (!allow_wide || !has_wide(D, G)) return G < kMmaMinGroup ? 2 : 1;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const long long stages = static_cast<long long>(B) * Hkv * ((max_ctx + 2 * kTN - 1) / (2 * kTN));
    return stages >= static_cast<long long>(kWideMinStagesPerSm) * device_sm_count() ? 2 : 1;
}

// Units of the dynamic tail a launch's workspace holds: for the kernels with one producer warp and
// batches of at most 32 CTAs' threads of sequences whose table could hold enough tiles per CTA (an
// upper bound: every sequence at the table's full length; the kernel decides on the real count);
// none when the caller's scratch is fixed (allow_dynamic false).
int tail_units_for(int B, int Hkv, int G, int D, int max_blocks_per_seq, int block_size, size_t P,
                   bool allow_dynamic) {
    if (!allow_dynamic || producers_for(D, G) != 1 || B > kDynCoarse * threads_for(D, G)) return 0;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const long long tiles = static_cast<long long>(B) * Hkv * ((max_ctx + kTN - 1) / kTN);
    if (tiles < static_cast<long long>(kDynMinTilesPerCta) * static_cast<long long>(P)) return 0;
    return static_cast<int>(P) * kTailUnitsPerCta;
}

// Workspace layout: partials [units][2][G][D + 2] floats, records [units], the tail's counter.
struct WsLayout {
    size_t part, rec, ctr, total;
};
WsLayout ws_layout(size_t units, int G, int D) {
    WsLayout w{};
    w.part = 0;
    w.rec = (units * 2 * G * (D + 2) * sizeof(float) + 255) / 256 * 256;
    w.ctr = w.rec + (units * sizeof(SegRecord) + 15) / 16 * 16;
    w.total = w.ctr + 16;
    return w;
}

// a distinct, non-zero number per launch (records and the tail's counter carry it)
unsigned next_epoch() {
    static std::atomic<unsigned> e{0};
    unsigned v = e.fetch_add(1u) + 1u;
    if (v == 0) v = e.fetch_add(1u) + 1u;
    return v;
}

}  // namespace

DecodePlan plan_decode(int B, int Hq, int Hkv, int D, int max_blocks_per_seq, int block_size,
                       bool allow_wide) {
    DecodePlan plan{};
    const int G = Hq / Hkv;
    const size_t P = static_cast<size_t>(device_sm_count()) *
                     launch_ctas_per_sm(B, Hq, Hkv, D, max_blocks_per_seq, block_size, allow_wide);
    const size_t units = P + tail_units_for(B, Hkv, G, D, max_blocks_per_seq, block_size, P, allow_wide);
    plan.ws_bytes = ws_layout(units, G, D).total;
    return plan;
}

int decode_debug_tail_units(const void *workspace, int B, int Hq, int Hkv, int D,
                            int max_blocks_per_seq, int block_size) {
    if (!workspace || B < 1 || Hkv < 1 || Hq % Hkv || max_blocks_per_seq < 1 || block_size < 1) return -1;
    const int G = Hq / Hkv;
    const size_t P = static_cast<size_t>(device_sm_count()) *
                     launch_ctas_per_sm(B, Hq, Hkv, D, max_blocks_per_seq, block_size, true);
    const size_t units = P + tail_units_for(B, Hkv, G, D, max_blocks_per_seq, block_size, P, true);
    // unit 0 is the static unit of CTA 0, whose record every launch writes
    SegRecord r{};
    const char *rec = static_cast<const char *>(workspace) + ws_layout(units, G, D).rec;
    if (cudaMemcpy(&r, rec, sizeof(r), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
    return r.K2;
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    // short contexts: one CTA per pair, a chain of two memory round trips (decode_short.cu)
    if (short_decode_supported(a)) return launch_decode_short(a, stream);
    DecodeParams prm{};
    // rows per TMA box: the largest power of two dividing both the block size and the tile
    int R = 1;
    while (R < kTN && a.block_size % (2 * R) == 0) R *= 2;
    const long long slots = static_cast<long long>(a.num_blocks) * a.block_size;
    const int G = a.Hq / a.Hkv;
    const bool sw = G >= kMmaMinGroup;  // tensor-core consumers read swizzled tiles
    if (!encode_pool_cached(&prm.tmap_k, a.k_cache, a.dtype, a.D, a.Hkv, slots, R, sw) ||
        !encode_pool_cached(&prm.tmap_v, a.v_cache, a.dtype, a.D, a.Hkv, slots, R, sw))
        return cudaErrorInvalidValue;
    prm.q = a.q;
    prm.k_new = a.k_new;
    prm.v_new = a.v_new;
    prm.k_cache = const_cast<void *>(a.k_cache);
    prm.v_cache = const_cast<void *>(a.v_cache);
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.out = a.out;
    const int cps = launch_ctas_per_sm(a.B, a.Hq, a.Hkv, a.D, a.max_blocks, a.block_size, a.allow_wide);
    const size_t P = static_cast<size_t>(device_sm_count()) * cps;
    prm.tail_units = tail_units_for(a.B, a.Hkv, G, a.D, a.max_blocks, a.block_size, P, a.allow_wide);
    const WsLayout w = ws_layout(P + prm.tail_units, G, a.D);
    if (w.total > plan.ws_bytes) return cudaErrorInvalidValue;  // the plan and the launch disagree
    char *ws = static_cast<char *>(a.workspace);
    prm.part = reinterpret_cast<float *>(ws + w.part);
    prm.rec = reinterpret_cast<SegRecord *>(ws + w.rec);
    prm.ctr = reinterpret_cast<unsigned long long *>(ws + w.ctr);
    prm.epoch = next_epoch();
    prm.err = a.err;
    prm.B = a.B;
    prm.Hq = a.Hq;
    prm.Hkv = a.Hkv;
    prm.max_blocks = a.max_blocks;
    prm.num_blocks = a.num_blocks;
    prm.box_rows = R;
    prm.geom.block_size = a.block_size;
    prm.geom.shift = log2_if_pow2(a.block_size);
    prm.scale_log2 = a.scale * kLog2e;
    const bool wide = cps == 2 && has_wide(a.D, G);
    if (a.D == 128)
        return a.dtype == PA_BF16 ? dispatch_group<128, BF16>(G, wide, prm, stream)
                                  : dispatch_group<128, F16>(G, wide, prm, stream);
    return a.dtype == PA_BF16 ? dispatch_group<64, BF16>(G, wide, prm, stream)
                              : dispatch_group<64, F16>(G, wide, prm, stream);
}

}  // namespace pa
