// fa_bwd_onepass.cuh — the one-pass backward kernel for sm_103a: dK, dV and
// dQ of exact attention with every (query tile, key tile) pair visited once.
//
// The gradients are those of fa_bwd_kernel.cuh ("Why FlashAttention Can
// Avoid a Square Attention Array Without Making Attention Linear", section
// "Backward can recreate tiles instead of retaining the square"): per pair
//   dV_j += P^T dO_i,  dP = dO_i V_j^T,  dS = P * (dP - D),
//   dK_j += scale dS^T Q_i,  dQ_i += scale dS K_j.
// A CTA owns key tile j (K_j, V_j resident in shared memory) and streams
// the query tiles past it, like the dK/dV pass of fa_bwd, and also forms
// dQ_i = dS K_j for every query tile it visits and adds it in fp32 into a
// workspace: five tile products per pair instead of seven, at the price of
// the fp32 additions (done by the TMA engine, in no fixed order).
//
// CTA layout (576 threads, 96 registers each): warps 0-15 do the
// element-wise work, warp w on TMEM lanes 32*(w%4) .. +31 and on the
// 32-query column block w/4 of each tile (four warps per lane quarter, so
// each SM sub-partition runs four element-wise warps); warp 16 issues the
// tcgen05 MMAs from one thread; warp 17 issues the TMA loads from one
// thread.  TMEM: S^T in columns 0-127, dP^T in 128-255, dV and dK
// from 256; dQ in the dP^T columns at d = 128 (TMEM is full) and in two
// buffers of its own at d = 64.
//
// Per query tile i the element-wise warps run three phases:
//   1  P^T = 2^(S^T c - LSE), written 16-bit over the S^T columns just read;
//   2  dS^T = P^T * (dP^T - D), written to a shared-memory dS tile that is A
//      of dK (K-major: keys x queries) and of dQ (MN-major: queries x keys);
//   3  dQ_i read from TMEM, staged as 32-row x 16-column fp32 blocks, one
//      per warp, which the TMA engine adds into the workspace.
// Phase 1 of tile i+1 runs between phases 2 and 3 of tile i, while the
// tensor core forms dK_j += dS^T Q_i and dQ_i.  The MMA thread issues, per
// tile: dV (after phase 1), S^T of the next tile, dK and dQ (after phase 2),
// then dP^T of the next tile (at d = 128 once phase 3 has read dQ).
//
// With dropout (kDrop) the mask of the forward pass is drawn once per pair
// from (seed, offset) exactly as fa_bwd_dropout draws it: dV_j += (P Z)^T dO_i
// (scaled by 256 / t at the end) and dS = P * (Z dP 256 / t - D).
#pragma once

#include "fa_bwd_kernel.cuh"
#include "fa_philox.cuh"

namespace fa {

constexpr int kOneThreads = 576;
constexpr int kOneEwThreads = 512;       // element-wise warps 0-15
constexpr int kOneMmaWarp = 16;
constexpr int kOneLoadWarp = 17;

// 32 lanes x 16 columns of 32 bits from this warp's lanes into 16 registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// One CTA of the one-pass backward: work item blk, one key tile of one head
// (dealt by bwd_item in groups of heads).  The fp32 dQ workspace (BwdParams::dq_acc) holds blocks of 32 queries x 16
// columns: block (bh, query tile qt, column block cb, row quarter rq) keeps
// element (column cc, row rr) at
//   dq_acc[((((bh * n_tiles + qt) * (D / 16) + cb) * 4 + rq) * 16 + cc) * 32 + rr].
template <int D, bool kBf16, bool kCausal, bool kDrop>
__device__ __forceinline__ void bwd_onepass_cta(const BwdParams& p, int blk, uint32_t tmem_base) {
  using L = BwdSmem<D, DkdvVec<D>::kBytes, true>;
  using X = DkdvBars;
  using Q = DqBuf<D>;
  static_assert(kOneEwThreads / 32 * 2048 <= L::kStgBytes, "staging blocks fit");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  auto xbar = [&](int i) -> uint32_t { return bar(L::bX + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kMisc + 4);

  // Key tile kt of head bh: items come in groups of item_group heads, key
  // tile by key tile within a group, so for causal runs the first key tiles
  // of a group (the most query tiles to visit) are dealt first.  Query
  // tiles i >= kt see key tile kt.
  int kt, bh;
  bwd_item(p, blk, p.n_ktiles, kt, bh);
  const int i0 = kCausal ? kt : 0;
  const int nq = p.n_tiles - i0;

  bwd_setup<L>(sbase, sgen, [&](auto b) {
    ptx::mbar_init(b(L::bX + X::kSFull), 1);
    ptx::mbar_init(b(L::bX + X::kDpFull), 1);
    ptx::mbar_init(b(L::bX + X::kPReady), kOneEwThreads);
    ptx::mbar_init(b(L::bX + X::kDsReady), kOneEwThreads);
    ptx::mbar_init(b(L::bX + X::kDone), 1);
    for (int q = 0; q < Q::kBufs; ++q) {
      ptx::mbar_init(b(L::bX + X::kDqFull + q), 1);
      ptx::mbar_init(b(L::bX + X::kDqFree + q), kOneEwThreads);
    }
  });
  const ptx::Watchdog wd{p.watchdog_cycles, abort_flag, p.status};

  if (warp == kOneLoadWarp) {
    if (lane == 0)
      bwd_producer<L>(sbase, &p.tm_k, &p.tm_v, kt, &p.tm_q, &p.tm_do, i0, nq, bh, wd);
    __syncwarp();
  } else if (warp == kOneMmaWarp) {
    if (lane == 0) {
      constexpr int fmt = kBf16 ? 1 : 0;
      constexpr uint32_t idesc_s = ptx::idesc_f16(kBwdTile, kBwdTile, fmt, 0);
      constexpr uint32_t idesc_acc = ptx::idesc_f16(kBwdTile, D, fmt, 1);   // dV, dK: B MN-major
      constexpr uint32_t idesc_dq = idesc_acc | kIdescAMnMajor;             // dQ: A MN-major too
      constexpr uint32_t kSlotLo = L::kTile >> 4;
      const uint32_t k_lo = ptx::desc_lo(sbase + L::kRes, 16);
      const uint32_t v_lo = ptx::desc_lo(sbase + L::kRes + L::kTile, 16);
      const uint32_t k_mn = ptx::desc_lo(sbase + L::kRes, L::kChunkBytes);
      const uint32_t q_lo0 = ptx::desc_lo(sbase + L::kRingA, 16);
      const uint32_t do_lo0 = ptx::desc_lo(sbase + L::kRingB, 16);
      const uint32_t q_mn0 = ptx::desc_lo(sbase + L::kRingA, L::kChunkBytes);
      const uint32_t do_mn0 = ptx::desc_lo(sbase + L::kRingB, L::kChunkBytes);
      const uint32_t ds_k = ptx::desc_lo(sbase + L::kDs, 16);
      const uint32_t ds_mn = ptx::desc_lo(sbase + L::kDs, L::kChunkBytes);
      const uint32_t tS = tmem_base + kColS, tDp = tmem_base + kColDp;
      const uint32_t tDv = tmem_base + kColAcc, tDk = tmem_base + kColAcc + D;
      auto full_a = [&](int it) {
        return ptx::wait_bounded(bar(L::bFullA + it % L::kStagesA), (it / L::kStagesA) & 1, wd,
                                 kSiteBwdFull);
      };
      auto full_b = [&](int it) {
        return ptx::wait_bounded(bar(L::bFullB + it % L::kStagesB), (it / L::kStagesB) & 1, wd,
                                 kSiteBwdFull);
      };
      // S^T = K_j Q_i^T and dP^T = V_j dO_i^T (keys on the TMEM lanes)
      auto issue_s = [&](int it) {
        issue_kmajor<D, L::kChunkBytes>(tS, k_lo, q_lo0 + (it % L::kStagesA) * kSlotLo, idesc_s);
        ptx::mma_commit(xbar(X::kSFull));
      };
      auto issue_dp = [&](int it) {
        issue_kmajor<D, L::kChunkBytes>(tDp, v_lo, do_lo0 + (it % L::kStagesB) * kSlotLo,
                                        idesc_s);
        ptx::mma_commit(xbar(X::kDpFull));
      };
      bool alive = ptx::wait_bounded(bar(L::bRes), 0, wd, kSiteBwdRes);
      alive = alive && full_a(0) && full_b(0);
      ptx::tc_fence_after();
      if (alive) {
        issue_s(0);
        issue_dp(0);
      }
      for (int it = 0; alive && it < nq; ++it) {
        const bool more = it + 1 < nq;
        alive = ptx::wait_bounded(xbar(X::kPReady), it & 1, wd, kSiteBwdPFull);
        ptx::tc_fence_after();
        if (!alive) break;
        // dV_j += P^T dO_i: P^T of queries 32c .. 32c + 31 sits, 16-bit, in
        // TMEM columns 32c .. 32c + 15
#pragma unroll
        for (int kk = 0; kk < kBwdTile / 16; ++kk)
          ptx::mma_ts(tDv, tS + (kk >> 1) * 32 + (kk & 1) * 8,
                      ptx::desc_sw128(do_mn0 + (it % L::kStagesB) * kSlotLo + kk * (2048 >> 4)),
                      idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar(L::bEmptyB + it % L::kStagesB));
        if (more) {
          alive = full_a(it + 1);
          ptx::tc_fence_after();
          if (!alive) break;
          issue_s(it + 1);   // after dV in this thread's order: P^T has been read
        }
        alive = ptx::wait_bounded(xbar(X::kDsReady), it & 1, wd, kSiteBwdDsReady);
        ptx::tc_fence_after();
        if (!alive) break;
        // dK_j += dS^T Q_i (scale applied at the end)
        issue_smem_a<L::kChunkBytes>(tDk, ds_k, q_mn0 + (it % L::kStagesA) * kSlotLo, idesc_acc,
                                     it > 0 ? 1u : 0u);
        ptx::mma_commit(bar(L::bEmptyA + it % L::kStagesA));
        // dQ_i = dS K_j into a dQ buffer the element-wise warps have emptied
        // (with one buffer, the dP^T columns: read before dS was ready)
        const int b = it % Q::kBufs;
        if (Q::kBufs > 1 && it >= Q::kBufs) {
          alive = ptx::wait_bounded(xbar(X::kDqFree + b), ((it / Q::kBufs) - 1) & 1, wd,
                                    kSiteBwdDqFree);
          ptx::tc_fence_after();
          if (!alive) break;
        }
        issue_mn_mn(tmem_base + Q::col(b), ds_mn, k_mn, idesc_dq);
        ptx::mma_commit(xbar(X::kDqFull + b));
        if (more) {
          alive = full_b(it + 1);
          if (Q::kBufs == 1)   // dP^T_{i+1} overwrites dQ_i: wait until it is read
            alive = alive && ptx::wait_bounded(xbar(X::kDqFree), it & 1, wd, kSiteBwdDqFree);
          ptx::tc_fence_after();
          if (!alive) break;
          issue_dp(it + 1);
        }
      }
      ptx::mma_commit(xbar(X::kDone));
      ptx::wait_drain(xbar(X::kDone), 0, 200000000ull);
    }
    __syncwarp();
  } else if (warp < kOneEwThreads / 32) {
    // ============================================================ element-wise
    ptx::griddep_wait();   // D of the pass launched just before this grid
    const int quarter = warp & 3, part = warp >> 2;
    const int t = quarter * 32 + lane;   // key row (phases 1, 2) or query row (phase 3)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // this thread's 32 query columns of S^T and dP^T
    const uint32_t tS = tmem_base + lane_off + kColS + part * 32;
    const uint32_t tDp = tmem_base + lane_off + kColDp + part * 32;
    const long long key = static_cast<long long>(kt) * kBwdTile + t;
    const uint64_t c2 = ptx::f2_pack(p.scale_log2, p.scale_log2);

    // LSE and D of query row t of tile i, fetched one tile ahead by the
    // warps of column block 0; the loads are unconditional (a row past the
    // queries reads row 0) and their values are used only when the tile is
    // staged, so no warp waits on them.  A query past N gets -LSE = -inf
    // (its P is 0) and D = 0.
    bool in_next = false;
    float lse_next = 0.f, d_next = 0.f;
    auto fetch = [&](int i) {
      const int qrow = i * kBwdTile + t;
      in_next = qrow < p.N;
      const long long qi = static_cast<long long>(bh) * p.N + (in_next ? qrow : 0);
      lse_next = p.lse[qi];
      d_next = p.delta[qi];
    };
    if (part == 0) fetch(i0);
    // vectors of query tile i0 + it: [0,128) -LSE in log2 units, [128,256) D
    auto vec_of = [&](int it) {
      return reinterpret_cast<float*>(sgen + L::kVec) + (it % DkdvVec<D>::kBufs) * 256;
    };
    auto stage_vec = [&](int it) {
      float* vec = vec_of(it);
      // with one buffer, every thread must be done with the previous tile's
      if (DkdvVec<D>::kBufs == 1 && it > 0) ptx::named_bar_sync(1, kOneEwThreads);
      if (part == 0) {
        vec[t] = in_next ? -lse_next * 1.4426950408889634f : -INFINITY;
        vec[128 + t] = in_next ? d_next : 0.f;
        if (it + 1 < nq) fetch(i0 + it + 1);
      }
      ptx::named_bar_sync(2, kOneEwThreads);
    };

    float pf[32];   // P^T of the current tile, from phase 1 to phase 2
    // dropout: the quad's words for this key block against the thread's 32
    // queries (zw[k2]: the word of quad lane k2), from phase 1 to phase 2;
    // zq(b) has byte r's top bit set when query 4b + r is kept
    uint32_t zw[4] = {0u, 0u, 0u, 0u};
    const uint32_t csel = 0x4440u + (static_cast<uint32_t>(lane) & 3u);   // this key's byte
    auto zq = [&](int b) -> uint32_t { return col_query_bits(zw[b & 3], csel, b >> 2); };
    auto phase1 = [&](int it) {
      const int i = i0 + it;
      const float4* nl4 = reinterpret_cast<const float4*>(vec_of(it)) + part * 8;
      ptx::wait_bounded(xbar(X::kSFull), it & 1, wd, kSiteBwdSFull);
      __syncwarp();
      ptx::tc_fence_after();
      uint32_t sr[32];
      ptx::tmem_ld32(tS, sr);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 nl = nl4[e / 4];
        float x0, x1, x2, x3;
        ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                  c2, ptx::f2_pack(nl.x, nl.y)), x0, x1);
        ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])),
                                  c2, ptx::f2_pack(nl.z, nl.w)), x2, x3);
        pf[e] = ptx::ex2(x0);
        pf[e + 1] = ptx::ex2(x1);
        pf[e + 2] = ptx::ex2(x2);
        pf[e + 3] = ptx::ex2(x3);
      }
      if (kCausal && i == kt) {   // diagonal tile: a key after the query is masked
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (i * kBwdTile + part * 32 + e < key) pf[e] = 0.f;
      }
      if constexpr (kDrop) {
        const uint32_t mine = drop_words8(static_cast<uint32_t>(key >> 2),
                                          static_cast<uint32_t>(i * kBwdTile + part * 32) >> 2,
                                          static_cast<uint32_t>(lane) & 3u,
                                          static_cast<uint32_t>(bh), p.drop_off, p.drop_k0,
                                          p.drop_k1, p.drop_t);
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) zw[k2] = __shfl_sync(0xffffffffu, mine, (lane & ~3) | k2);
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        pk[e] = ptx::pack2<kBf16>(pf[2 * e], pf[2 * e + 1]);
        // the dV product reads P with the dropped weights zeroed
        if constexpr (kDrop) pk[e] &= prmt(zq(e >> 1), 0u, (e & 1) ? 0xBBAAu : 0x9988u);
      }
      ptx::tmem_st16(tS, pk);   // over the S^T columns this warp has read
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(xbar(X::kPReady));
    };

    auto phase2 = [&](int it) {
      const float4* dl4 = reinterpret_cast<const float4*>(vec_of(it) + 128) + part * 8;
      ptx::wait_bounded(xbar(X::kDpFull), it & 1, wd, kSiteBwdDpFull);
      __syncwarp();
      ptx::tc_fence_after();
      uint32_t dpr[32];
      ptx::tmem_ld32(tDp, dpr);
      ptx::tmem_wait_ld();
      uint32_t ds[16];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 dd = dl4[e / 4];
        // dP^T, with dropout Z dP^T (the 256 / t joins in the subtraction of D)
        uint32_t zx = 0;
        if constexpr (kDrop) zx = zq(e >> 2);   // e is a multiple of 4: one block
        auto dpv = [&](int x) -> float {
          if constexpr (kDrop)
            return __uint_as_float(dpr[e + x] & prmt(zx, 0u, 0x8888u + 0x1111u * x));
          return __uint_as_float(dpr[e + x]);
        };
        auto dmd = [&](float a, float b, float da, float db) -> uint64_t {
          if constexpr (kDrop)
            return ptx::ffma2(ptx::f2_pack(a, b), ptx::f2_pack(p.drop_scale, p.drop_scale),
                              ptx::f2_pack(-da, -db));
          return ptx::fadd2(ptx::f2_pack(a, b), ptx::f2_pack(-da, -db));
        };
        float d0, d1, d2, d3;
        ptx::f2_unpack(ptx::fmul2(ptx::f2_pack(pf[e], pf[e + 1]), dmd(dpv(0), dpv(1), dd.x, dd.y)),
                       d0, d1);
        ptx::f2_unpack(ptx::fmul2(ptx::f2_pack(pf[e + 2], pf[e + 3]),
                                  dmd(dpv(2), dpv(3), dd.z, dd.w)), d2, d3);
        ds[e / 2] = ptx::pack2<kBf16>(d0, d1);
        ds[e / 2 + 1] = ptx::pack2<kBf16>(d2, d3);
      }
      // row t (key) of the dS tile: this thread's 32 queries are 16-byte
      // pieces 4 (part % 2) .. + 3 of query chunk part / 2, in the 128-byte
      // swizzle (the previous tile's dK and dQ, which read the tile,
      // completed before this warp's phase 3 of that tile went on)
      uint8_t* drow = sgen + L::kDs + (part >> 1) * L::kChunkBytes + t * 128;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int c = (part & 1) * 4 + c4;
        *reinterpret_cast<uint4*>(drow + ((c ^ (t & 7)) << 4)) =
            make_uint4(ds[4 * c4], ds[4 * c4 + 1], ds[4 * c4 + 2], ds[4 * c4 + 3]);
      }
      ptx::fence_proxy_async_smem();   // visible to the tensor core's reads
      ptx::tc_fence_before();
      ptx::mbar_arrive(xbar(X::kDsReady));
    };

    // phase 3: dQ_i (queries on the TMEM lanes; this thread: query row t,
    // columns part * D/4 .. + D/4) to the workspace
    constexpr int kCw = D / 4;
    float* stg = reinterpret_cast<float*>(sgen + L::kStg + warp * 2048);
    const uint32_t stg_s = sbase + L::kStg + warp * 2048;
    auto phase3 = [&](int it) {
      const int i = i0 + it;
      const int b = it % Q::kBufs;
      ptx::wait_bounded(xbar(X::kDqFull + b), (it / Q::kBufs) & 1, wd, kSiteBwdDqFull);
      __syncwarp();
      ptx::tc_fence_after();
      const uint32_t tq = tmem_base + lane_off + Q::col(b) + part * kCw;
      uint32_t r[kCw];
      if constexpr (kCw == 32) {
        ptx::tmem_ld32(tq, r);
      } else {
        tmem_ld16(tq, r);
      }
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(xbar(X::kDqFree + b));   // the buffer may be overwritten now
#pragma unroll
      for (int k = 0; k < kCw / 16; ++k) {
        if (lane == 0) bulk_wait_read_all();   // the block's previous contents are sent
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) stg[cc * 32 + lane] = __uint_as_float(r[k * 16 + cc]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int cb = part * (kCw / 16) + k;
          const long long blk =
              ((static_cast<long long>(bh) * p.n_tiles + i) * (D / 16) + cb) * 4 + quarter;
          bulk_reduce_add_f32(p.dq_acc + blk * 512, stg_s, 2048);
        }
      }
    };

    // Phase 1 of the next tile runs while the tensor core forms this tile's
    // dK and dQ; phase 3 then finds dQ ready.
    stage_vec(0);
    phase1(0);
    for (int it = 0; it < nq; ++it) {
      phase2(it);
      if (it + 1 < nq) {
        stage_vec(it + 1);
        phase1(it + 1);
      }
      phase3(it);
    }
    if (lane == 0) bulk_wait_all();   // this warp's dQ additions have landed
    __syncwarp();
    // dV_j (column blocks 0, 1) and dK_j = scale * (dS^T Q) (2, 3): each warp
    // stores half of the columns of its 32 key rows
    ptx::wait_bounded(xbar(X::kDone), 0, wd, kSiteBwdDone);
    __syncwarp();
    ptx::tc_fence_after();
    const long long row = static_cast<long long>(bh) * p.Nk + key;
    const int c0 = (part & 1) * (D / 2);
    if (part < 2)
      store_acc_cols<kBf16>(tmem_base + lane_off + kColAcc, c0, D / 2, D,
                            kDrop ? p.drop_scale : 1.f, p.dv, row, key < p.Nk);
    else
      store_acc_cols<kBf16>(tmem_base + lane_off + kColAcc + D, c0, D / 2, D, p.scale, p.dk, row,
                            key < p.Nk);
  }
  bwd_teardown<L>(sbase);
}

// The one-pass backward grid: at most one CTA per SM walking the key tiles
// (the ones with the most query tiles first); the CTA allocates TMEM once.
template <int D, bool kBf16, bool kCausal, bool kDrop = false>
__global__ void __launch_bounds__(kOneThreads, 1)
    fa_bwd_onepass_kernel(const __grid_constant__ BwdParams p) {
  __shared__ uint32_t s_tmem_base;
  const int warp = threadIdx.x >> 5;
  if (warp == kOneMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem_base), kBwdTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int items = p.BH * p.n_ktiles;
  for (int item = blockIdx.x; item < items; item += gridDim.x)
    bwd_onepass_cta<D, kBf16, kCausal, kDrop>(p, item, tmem_base);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kOneMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kBwdTmemCols);
  }
}

}  // namespace fa
