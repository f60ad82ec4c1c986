// Exact attention forward for head dim 256 (sm_103a).
//
// At D = 256 an O accumulator takes 256 of the 512 tensor-memory columns, so
// a CTA holds ONE 128-row query tile per unit (the D <= 128 kernel holds two):
//   tensor memory  S_even [0, 128)   O [128, 384)   S_odd [384, 512)
// and both softmax warpgroups work on that tile's rows: warpgroup w owns score
// columns [64 w, 64 w + 64) (keys of the K/V tile) and O columns
// [128 w, 128 w + 128).  The scores of K/V tiles j and j + 1 go to different
// buffers, so the MMA thread issues S(j + 1) = Q K(j + 1)^T before O += P(j)
// V(j) and the tensor pipe works on it while the softmax works on S(j):
//   S(0) S(1) | PV(0) S(2) | PV(1) S(3) | ...
// (one tile per unit has no second tile to alternate with).  A rescale of O at
// tile j waits until O += P(j - 1) V(j - 1) has completed (pv_done).  Per K/V
// tile j:
//   * each warpgroup loads its half of S_j, takes its half-row max and hands it
//     to the other through shared memory (named barrier 3 over 256 threads);
//     both then hold the same row max and take the same lazy-rescale decision
//     (threshold 8 log2 units, max lagging, first tile sets the max), so each
//     rescales its own half of O and its own partial row sum;
//   * warpgroup w writes P of its 64 keys as 16-bit pairs into columns
//     [32 w, 32 w + 32) of the tile's score buffer and signals p_half[b][w]
//     of that buffer b (the softmax may finish tile j + 1, whose scores are
//     ready early, before O += P(j) V(j) is issued: full / ready barriers per
//     buffer keep the phases of consecutive tiles apart);
//     warpgroup 1 writes only after the barrier, i.e. after warpgroup 0 has
//     read its S columns 32-63;
//   * one MMA thread issues O += P V in two halves (keys 0-63 as soon as
//     warpgroup 0's P is stored, keys 64-127 after warpgroup 1's), each four
//     M128 N256 K16 steps with P straight from tensor memory, then
//     S = Q K(j+2)^T into the same buffer as sixteen M128 N128 K16 steps (the
//     tensor pipe runs one CTA's MMAs in issue order, so that S is written
//     after P(j) has been read).
// The K/V ring holds two 64 KB tiles, loaded in the order the MMAs read them:
// K(0), K(1), V(0), K(2), V(1), ..., K(n-1), V(n-2), V(n-1).  The epilogue adds the
// two partial row sums through shared memory; each warpgroup normalises and
// stores its 128 columns of O.  For packed sequences warp 10 zeroes the V rows
// of a unit's last K/V tile that lie past the sequence's last key (they hold
// the next sequence's data) before that tile is used.
#pragma once

#include "fa_launch.cuh"

namespace fa {

// 384 threads: two softmax warpgroups and one control warpgroup.
constexpr int kWideThreads = 384;

template <int D>
struct SmemWide {
  static constexpr int kChunks = D / 64;                     // 64-element swizzle chunks
  static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = D == 256 ? 2 : 8;           // K/V ring depth
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = kTileBytes;
  // output staging for the TMA store, 128 rows x kStoreCols columns per
  // warpgroup (128B swizzle for 64 columns, 64B for 32)
  static constexpr int kStoreCols = D / 2 < 64 ? D / 2 : 64;
  static constexpr uint32_t kStageBytes = 128u * kStoreCols * 2u;
  static constexpr uint32_t kStageOff = kKVOff + kStages * kTileBytes;
  // half-row maxima / partial row sums exchanged between the warpgroups
  static constexpr uint32_t kXchOff = kStageOff + 2 * kStageBytes;
  static constexpr uint32_t kBarOff = kXchOff + 2 * 128 * 4;
  // barriers: q_full, q_empty, kv_full[S], kv_empty[S], p_half[2][2], o_ready,
  //           o_free, drain, v_fixed[S], s_full[2], pv_done (S = kStages)
  static constexpr int kNumBars = 12 + 3 * kStages;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kBytes = kMiscOff + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

template <int D, bool BF16, bool CAUSAL, bool VARLEN, bool EXT>
__global__ void __launch_bounds__(kWideThreads, 1)
    fa_fwd_wide_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  static_assert(D == 64 || D == 256, "single-tile kernel: head dim 64 or 256");
  constexpr int DH = D / 2;  // O columns of one warpgroup
  using L = SmemWide<D>;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBarOff;
  const uint32_t q_full = bar0, q_empty = bar0 + 8;
  // barrier indices: q_full 0, q_empty 1, kv_full [2, 2 + S), kv_empty
  // [2 + S, 2 + 2S), p_half [2 + 2S, 6 + 2S), o_ready, o_free, drain,
  // v_fixed [9 + 2S, 9 + 3S), s_full [9 + 3S, 11 + 3S), pv_done (S = ring stages)
  constexpr int S = L::kStages;
  auto kv_full = [&](int s) { return bar0 + 8u * (2 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (2 + S + s); };
  // score buffer b is full / holds P of keys [64 h, 64 h + 64)
  auto s_full = [&](int b) { return bar0 + 8u * (9 + 3 * S + b); };
  auto p_half = [&](int b, int h) { return bar0 + 8u * (2 + 2 * S + 2 * b + h); };
  const uint32_t o_ready = bar0 + 8u * (6 + 2 * S), o_free = bar0 + 8u * (7 + 2 * S);
  const uint32_t drain_bar = bar0 + 8u * (8 + 2 * S);
  auto v_fixed = [&](int s) { return bar0 + 8u * (9 + 2 * S + s); };
  const uint32_t pv_done = bar0 + 8u * (11 + 3 * S);  // O += P(j) V(j) has completed
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
  // K/V loads the producer has issued (the V-row fixer never waits a lap ahead)
  volatile int *kv_issued = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 8);
  float *xch = reinterpret_cast<float *>(smem + L::kXchOff);  // [2][128]
  static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
      mbar_init(v_fixed(s), 1);
    }
    *kv_issued = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_half(b, 0), 4);  // one arrival per softmax warp of the half
      mbar_init(p_half(b, 1), 4);
    }
    mbar_init(o_ready, 1);
    mbar_init(o_free, 8);     // every softmax warp has read its O columns
    mbar_init(drain_bar, 1);
    mbar_init(pv_done, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const long long limit = p.wait_limit;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return wait_bar(bar, par, abort_flag, limit, p.status);
  };

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
    if (warp == kTmaWarp) {
      // ---------------------------------------------------------- TMA producer
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      int issued = 0, q_loads = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int unit = unit_of(i);
        if (unit >= p.total_units) break;
        const Work w = decode_work<CAUSAL, VARLEN, EXT, true>(p, unit, lane);
        if (!w.valid || w.n_kv[0] == 0) continue;
        if (lane == 0) {
          // the previous unit's Q is free once its last S = Q K^T is done
          if (q_loads > 0 && !wait(q_empty, (q_loads - 1) & 1)) {
            ok = false;
          } else {
            mbar_arrive_expect_tx(q_full, L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_4d(sbase + L::kQOff + c * kChunkBytes, &tm_q, q_full, c * 64, w.head[0],
                          w.q_row0 + w.m0[0], w.map_b, pol_q);
            ++q_loads;
          }
          // one K or V tile (which: 0 K, 1 V) of unit tile j into the next slot
          auto issue = [&](int which, int j) {
            const int idx = issued, s = idx % L::kStages;
            if (idx >= L::kStages && !wait(kv_empty(s), ((idx / L::kStages) + 1) & 1)) {
              ok = false;
              return;
            }
            mbar_arrive_expect_tx(kv_full(s), L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_4d(sbase + L::kKVOff + s * L::kTileBytes + c * kChunkBytes,
                          which == 0 ? &tm_k : &tm_v, kv_full(s), c * 64, w.hkv,
                          w.k_row0 + (w.kv_begin[0] + j) * kBlockN, w.map_b, pol_kv);
            issued = idx + 1;
            *kv_issued = issued;
          };
          // K runs one tile ahead of V: K(0), K(1), V(0), K(2), V(1), ...
          const int n = w.n_kv[0];
          if (ok) issue(0, 0);
          for (int j = 0; j < n && ok; ++j) {
            if (j + 1 < n) issue(0, j + 1);
            if (ok) issue(1, j);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (!ok && lane == 0) {
        // drain copies still in flight before the CTA exits
        for (int idx = max(0, issued - L::kStages); idx < issued; ++idx)
          wait_bar(kv_full(idx % L::kStages), (idx / L::kStages) & 1, abort_flag, limit,
                   p.status, false);
        if (q_loads > 0) wait_bar(q_full, (q_loads - 1) & 1, abort_flag, limit, p.status, false);
      }
    } else if (warp == kMmaWarp) {
      // --------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, kBlockM, kBlockN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, kBlockM, D, true);
      const uint64_t q_desc = make_sdesc_sw128(sbase + L::kQOff, 16, 1024);
      const uint64_t kv_desc0 = make_sdesc_sw128(sbase + L::kKVOff, 16, 1024);
      const uint64_t v_desc0 = make_sdesc_sw128(sbase + L::kKVOff, kChunkBytes, 1024);
      // score buffer of unit tile j: columns [0, 128) for even j, [384, 512) for odd j
      auto d_s = [&](int j) { return tmem + ((j & 1) ? 384u : 0u); };
      const uint32_t d_o = tmem + 128;
      auto issue_qk = [&](int kidx, uint32_t ds) {
        const uint64_t kd = kv_desc0 + (((kidx % L::kStages) * L::kTileBytes) >> 4);
        mma_ss(ds, q_desc, kd, idesc_qk, 0u);
#pragma unroll
        for (int kk = 1; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_acc(ds, q_desc + off, kd + off, idesc_qk);
        }
      };
      // O += P V for keys [64 h, 64 h + 64): P from buffer columns [32 h, 32 h + 32)
      auto issue_pv_half = [&](int vidx, uint32_t ds, int h, bool first) {
        const uint64_t vd = v_desc0 + (((vidx % L::kStages) * L::kTileBytes + h * 4 * 2048) >> 4);
        const uint32_t a = ds + h * 32;
        if (h == 0)
          mma_ts(d_o, a, vd, idesc_pv, first ? 0u : 1u);
        else
          mma_ts_acc(d_o, a, vd, idesc_pv);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk)
          mma_ts_acc(d_o, a + kk * 8, vd + ((kk * 2048) >> 4), idesc_pv);
      };
      auto kv_par = [&](int idx) { return (uint32_t)((idx / L::kStages) & 1); };
      int used = 0, q_used = 0, o_done = 0;
      int p_seen0 = 0, p_seen1 = 0;  // P tiles consumed per score buffer
      uint32_t vpar = 0;  // bit s: phase parity of v_fixed(s)
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int unit = unit_of(i);
        if (unit >= p.total_units) break;
        const Work w = decode_work<CAUSAL, VARLEN, EXT, true>(p, unit, lane);
        const int n = w.n_kv[0];
        if (!w.valid || n == 0) continue;
        // the unit's last V tile has rows past the sequence's keys: wait
        // until the fixer warp has zeroed them
        const bool vfix = v_tail_rows<VARLEN, false>(w) > 0;
        const int fix_idx = vfix ? used + 2 * n - 1 : -1;
        const int fix_slot = vfix ? fix_idx % L::kStages : 0;
        const uint32_t fix_par = (vpar >> fix_slot) & 1u;
        if (vfix) vpar ^= 1u << fix_slot;
        if (lane == 0) {
          // ring positions of the unit's loads (K one tile ahead of V)
          auto kpos = [&](int j) { return used + (j == 0 ? 0 : 2 * j - 1); };
          auto vpos = [&](int j) { return used + (j + 1 < n ? 2 * j + 2 : 2 * n - 1); };
          // S(j) = Q K(j)^T into buffer j % 2
          auto issue_s = [&](int j) {
            if (j == 0) {
              ok = wait(q_full, q_used & 1);
              ++q_used;
            }
            const int kidx = kpos(j);
            ok = ok && wait(kv_full(kidx % L::kStages), kv_par(kidx));
            if (!ok) return;
            tc_fence_after();
            issue_qk(kidx, d_s(j));
            tc_commit(s_full(j & 1));
            if (j == n - 1) tc_commit(q_empty);  // last S of this unit issued
            tc_commit(kv_empty(kidx % L::kStages));
          };
          issue_s(0);
          if (n > 1 && ok) issue_s(1);
          for (int j = 0; j < n && ok; ++j) {
            // O += P(j) V(j); the unit's first one overwrites O, which the
            // previous unit's epilogue must have read out
            const int vidx = vpos(j), b = j & 1;
            int &p_seen = b ? p_seen1 : p_seen0;
            ok = wait(kv_full(vidx % L::kStages), kv_par(vidx)) &&
                 (vidx != fix_idx || wait(v_fixed(fix_slot), fix_par)) &&
                 (j > 0 || o_done == 0 || wait(o_free, (o_done - 1) & 1)) &&
                 wait_bar_spin(p_half(b, 0), p_seen & 1, abort_flag, limit, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_pv_half(vidx, d_s(j), 0, j == 0);
            if (!wait_bar_spin(p_half(b, 1), p_seen & 1, abort_flag, limit, p.status)) {
              ok = false;
              break;
            }
            ++p_seen;
            tc_fence_after();
            issue_pv_half(vidx, d_s(j), 1, false);
            tc_commit(pv_done);
            if (j == n - 1) {
              tc_commit(o_ready);
              ++o_done;
            }
            tc_commit(kv_empty(vidx % L::kStages));
            // S(j + 2) reuses this buffer: the pipe runs it after P(j) is read
            if (j + 2 < n) issue_s(j + 2);
          }
          used += 2 * n;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (lane == 0) {
        // no MMA may still be running when tensor memory is released
        tc_commit(drain_bar);
        wait_bar(drain_bar, 0, abort_flag, limit, p.status, false);
      }
    } else if (warp == 10 && VARLEN) {
      // ------------------------------------------------- V rows past the keys
      // (see the D <= 128 kernel): zero the rows of a unit's last V tile past
      // the sequence's last key once it has landed, then signal v_fixed
      int used = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int unit = unit_of(i);
        if (unit >= p.total_units) break;
        const Work w = decode_work<CAUSAL, VARLEN, EXT, true>(p, unit, lane);
        const int n = w.n_kv[0];
        if (!w.valid || n == 0) continue;
        const int valid = v_tail_rows<VARLEN, false>(w);
        if (valid > 0) {
          const int idx = used + 2 * n - 1;  // ring index of the unit's last V load
          const int s = idx % L::kStages;
          const long long t0 = clock64();
          while (ok && *kv_issued <= idx) {
            __nanosleep(256);  // far ahead of the load: sleep, keep issue slots free
            if (*abort_flag) ok = false;
            if (clock64() - t0 > limit) {
              record_status(p.status, 4);
              *abort_flag = 1;
              ok = false;
            }
          }
          ok = __all_sync(0xffffffffu, ok && wait(kv_full(s), (idx / L::kStages) & 1));
          if (ok) {
            const uint32_t tile = sbase + L::kKVOff + s * L::kTileBytes;
#pragma unroll 1
            for (int c = 0; c < L::kChunks; ++c)
#pragma unroll 1
              for (uint32_t b = (uint32_t)valid * 128u + lane * 16u; b < kChunkBytes; b += 512u)
                st_shared_v4(tile + c * kChunkBytes + b, 0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(v_fixed(s));
          }
        }
        used += 2 * n;
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // ------------------------------------------------------ softmax + epilogue
    const int wg = warp >> 2;       // column half of this warpgroup
    const int quarter = warp & 3;   // TMEM lane quarter
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    // this half's score / P columns in the buffer of unit tile j, O columns
    auto s_addr = [&](int j) { return lane_base + ((j & 1) ? 384u : 0u) + wg * 64; };
    auto p_addr = [&](int j) { return lane_base + ((j & 1) ? 384u : 0u) + wg * 32; };
    const uint32_t o_addr = lane_base + 128 + wg * DH;
    const float scale_log2 = EXT ? 1.f : p.scale_log2;
    const float neg_thr = -p.threshold;
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
      const bool got = wait(bar, parity);
      return __all_sync(0xffffffffu, got);
    };
    float *x_mine = xch + wg * 128, *x_other = xch + (1 - wg) * 128;
    int s_seen0 = 0, s_seen1 = 0, o_seen = 0;  // score tiles consumed per buffer
    int pv_base = 0;  // O += P V products of earlier units (pv_done phases)
    const bool elected = quarter == 0 && lane == 0;
    const uint32_t stage = sbase + L::kStageOff + wg * L::kStageBytes;
    // Both warpgroups meet at named barrier 3 every K/V tile and twice per
    // unit; like the other kernel, the role never leaves its unit loop early.
    bool ok = true;
    for (int i = 0;; ++i) {
      const int unit = unit_of(i);
      if (unit >= p.total_units) break;
      const Work w = decode_work<CAUSAL, VARLEN, EXT, true>(p, unit, lane);
      if (!w.valid || w.m0[0] >= w.lq) continue;
      const int m0 = w.m0[0], n_kv = w.n_kv[0];
      const int lq = w.lq, lk = w.lk;
      const int qi = m0 + row;
      const int head = w.head[0];
      const int diag = qi + lk - lq;
      [[maybe_unused]] const float slope_l2 =
          (EXT && p.alibi) ? p.alibi[head] * 1.4426950408889634f : 0.f;
      float m = -INFINITY, l = 0.f;  // row max (shared), partial row sum (this half)
      for (int j = 0; j < n_kv; ++j) {
        int &s_seen = (j & 1) ? s_seen1 : s_seen0;
        bool got = ok && warp_wait(s_full(j & 1), s_seen & 1);
        ++s_seen;
        float s[64];
        if (got) {
          tc_fence_after();
          uint32_t sr[32];
          tmem_ld32(s_addr(j), sr);
          tmem_wait_ld32(sr);
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(sr[c]);
          tmem_ld32(s_addr(j) + 32, sr);
          tmem_wait_ld32(sr);
#pragma unroll
          for (int c = 0; c < 32; ++c) s[32 + c] = __uint_as_float(sr[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = -INFINITY;
        }
        const int k0 = (w.kv_begin[0] + j) * kBlockN + wg * 64;  // first key of this half
        if constexpr (EXT) {
          if (p.cap_k != 0.f) {
            soft_cap<64, true>(s, p.cap_k, p.cap_l2);
          } else {
            const float sl2 = p.scale_log2;
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] *= sl2;
          }
          if (p.alibi) {
            const float d0 = (float)(diag - k0);
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = fmaf(-slope_l2, fabsf(d0 - (float)c), s[c]);
          }
          const int lo = p.win_l < 0 ? -kBlockN : diag - p.win_l - k0;
          const int hi = min(lk, p.win_r < 0 ? lk : diag + p.win_r + 1) - k0;
          if (lo > 0 || hi < 64) {
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = (c >= lo && c < hi) ? s[c] : -INFINITY;
          }
        } else {
          int lim = lk - k0;
          if (CAUSAL) lim = min(lim, diag - k0 + 1);
          if (lim < 64) {
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
          }
        }
        // half-row max, exchanged with the other warpgroup
        const float hm = fmaxf(max32(s), max32(s + 32));
        x_mine[row] = hm;
        tc_fence_before();
        named_barrier_sync(3, 256);
        tc_fence_after();
        const float bm = fmaxf(hm, x_other[row]);
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m = bm;
        } else {
          const float m_cur = fmaxf(m, bm);
          const float diff = (m_cur == -INFINITY) ? 0.f : (m - m_cur) * scale_log2;
          if (!(diff >= neg_thr)) {
            alpha = ex2(diff);
            m = m_cur;
            rescale = true;
          }
        }
        if (got && __any_sync(0xffffffffu, rescale)) {
          // O += P(j-1) V(j-1), issued after S(j), may still be running: wait
          // until it has completed.  S(j) has completed, so P(j-2) V(j-2) has
          // too, and the parity names the product's phase unambiguously.
          l *= alpha;
          if (warp_wait(pv_done, (pv_base + j - 1) & 1)) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
              uint32_t orr[32];
              tmem_ld32_wait(o_addr + c * 32, orr);
#pragma unroll
              for (int k = 0; k < 32; ++k)
                orr[k] = __float_as_uint(__uint_as_float(orr[k]) * alpha);
              tmem_st32(o_addr + c * 32, orr);
            }
          } else {
            got = false;
            ok = false;
          }
        } else if (rescale) {
          l *= alpha;
        }
        const float ms = (m == -INFINITY) ? 0.f : m * scale_log2;
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        if (got) {
          softmax_chunk<BF16>(s, scale_log2, ms, acc, p_addr(j));
          softmax_chunk<BF16>(s + 32, scale_log2, ms, acc, p_addr(j) + 16);
          tmem_st_wait();
          tc_fence_before();
        }
        __syncwarp();
        if (got && lane == 0) mbar_arrive(p_half(j & 1, wg));
        if (!got) ok = false;
        add_f32x2(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        add_f32x2(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
        add_f32x2(acc[0].x, acc[0].y, acc[2].x, acc[2].y);
        l += acc[0].x + acc[0].y;
      }
      pv_base += n_kv;
      // ------------------------------------------------------------- epilogue
      uint32_t orr[DH];
#pragma unroll
      for (int k = 0; k < DH; ++k) orr[k] = 0u;
      if (n_kv > 0 && ok) {
        ok = warp_wait(o_ready, o_seen & 1);
        ++o_seen;
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < DH / 32; ++c)
            tmem_ld32(o_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(orr + 32 * c));
#pragma unroll
          for (int c = 0; c < DH / 32; ++c)
            tmem_wait_ld32(*reinterpret_cast<uint32_t(*)[32]>(orr + 32 * c));
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);
      }
      // full row sum: this half's plus the other's
      x_mine[row] = l;
      named_barrier_sync(3, 256);
      const float l_row = l + x_other[row];
      named_barrier_sync(3, 256);  // exchange buffer free for the next unit
      const float inv_l = l_row > 0.f ? 1.f / l_row : 0.f;
      const bool row_valid = qi < lq;
      const int64_t tok = w.o_row0 + qi;
      auto packed = [&](int k) {
        return pack_p<BF16>(__uint_as_float(orr[2 * k]) * inv_l,
                            __uint_as_float(orr[2 * k + 1]) * inv_l);
      };
      const int64_t li = VARLEN ? (int64_t)head * p.Sq + tok
                                : ((int64_t)w.b * p.Hq + head) * p.Sq + qi;
      const float lse = (l_row > 0.f) ? (m * scale_log2 + log2f(l_row)) * 0.69314718055994531f
                                      : -INFINITY;
      const bool use_tma = !VARLEN || (m0 + kBlockM <= lq);
      if (EXT && p.num_splits > 1) {
        if (row_valid && ok) {
          const int64_t slot = (int64_t)w.split * p.part_rows + li;
          float4 *dst = reinterpret_cast<float4 *>(p.o_part + slot * D + wg * DH);
#pragma unroll
          for (int k = 0; k < DH / 4; ++k)
            dst[k] = make_float4(__uint_as_float(orr[4 * k]) * inv_l,
                                 __uint_as_float(orr[4 * k + 1]) * inv_l,
                                 __uint_as_float(orr[4 * k + 2]) * inv_l,
                                 __uint_as_float(orr[4 * k + 3]) * inv_l);
          if (wg == 0) p.lse_part[slot] = lse;
        }
      } else if (use_tma) {
        constexpr int kSC = L::kStoreCols;
#pragma unroll
        for (int half = 0; half < DH / kSC; ++half) {
          named_barrier_sync(1 + wg, 128);  // staging buffer free
          if (ok) {
            // row `row`, 16-byte chunk c at its swizzled position: 128B
            // swizzle (64 columns) c ^ (row % 8), 64B swizzle (32 columns)
            // c ^ ((row / 2) % 4)
#pragma unroll
            for (int c = 0; c < kSC / 8; ++c) {
              const int k = half * (kSC / 2) + 4 * c;
              const int sc = kSC == 64 ? (c ^ (row & 7)) : (c ^ ((row >> 1) & 3));
              st_shared_v4(stage + row * (kSC * 2) + (sc << 4), packed(k), packed(k + 1),
                           packed(k + 2), packed(k + 3));
            }
            fence_proxy_async_smem();
          }
          named_barrier_sync(1 + wg, 128);  // staging buffer full
          if (elected) {
            if (ok) {
              tma_store_4d(&tm_o, stage, wg * DH + half * kSC, head, w.q_row0 + m0, w.map_b);
              bulk_commit_group();
            }
            bulk_wait_group_read0();
          }
        }
      } else if (row_valid && ok) {
        elem_t *o = reinterpret_cast<elem_t *>(p.o) + (tok * p.Hq + head) * (int64_t)D + wg * DH;
        uint4 *dst = reinterpret_cast<uint4 *>(o);
#pragma unroll
        for (int k = 0; k < DH / 8; ++k)
          dst[k] = make_uint4(packed(4 * k), packed(4 * k + 1), packed(4 * k + 2), packed(4 * k + 3));
      }
      if (wg == 0 && row_valid && ok && p.lse != nullptr && !(EXT && p.num_splits > 1))
        p.lse[li] = lse;
    }
    if (elected) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN, bool EXT>
cudaError_t launch_wide(const LaunchArgs &a) {
  auto kern = fa_fwd_wide_kernel<D, BF16, CAUSAL, VARLEN, EXT>;
  static SmemOptIn opt_in;
  const cudaError_t e = opt_in.ensure(kern, (int)SmemWide<D>::kAlloc, a.device, 168);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, kWideThreads, SmemWide<D>::kAlloc, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o,
                                                                 a.p);
  return cudaGetLastError();
}

}  // namespace fa
