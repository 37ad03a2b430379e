// fa_api.cu — the backward and decoding entry points of the C ABI declared
// in include/fa.h: argument checks, TMA descriptors and the launches of the
// backward and split-KV decoding kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "fa.h"
#include "fa_bwd_launch.cuh"
#include "fa_decode_kernel.cuh"
#include "fa_host.cuh"

using namespace fa::host;

extern "C" {

// Bytes of the one-pass backward's fp32 dQ accumulator: [B*H, d, N rounded
// up to whole 128-row tiles].
static long long onepass_acc_bytes(long long bh, long long n, int d) {
  const long long pad = (n + fa::kBwdTile - 1) / fa::kBwdTile * fa::kBwdTile;
  return bh * d * pad * static_cast<long long>(sizeof(float));
}

// fa_bwd, fa_bwd_dropout when drop_t < 256, fa_bwd_kv when kv (Nq queries
// against Nk keys with per-batch key counts; causal 2 bottom-right; values
// of width dv_width, which only kv calls may set apart from d), and
// fa_bwd_onepass when `one` (square calls; ws holds the dQ accumulator).
static int backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H,
                    int Nq, int Nk, int d, int dv_width, int causal, bool kv,
                    const int* seqlens_k, float scale, int dtype, int drop_t,
                    unsigned long long seed, unsigned int drop_off, cudaStream_t stream,
                    bool one = false, void* ws = nullptr, size_t ws_bytes = 0) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0 || dv_width <= 0) return FA_ERR_SHAPE;
  if (causal < 0 || causal > (kv ? 2 : 1)) return FA_ERR_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qtiles = (static_cast<long long>(Nq) + fa::kBwdTile - 1) / fa::kBwdTile;
  const long long n_ktiles = (static_cast<long long>(Nk) + fa::kBwdTile - 1) / fa::kBwdTile;
  if (bh > INT_MAX || bh * (n_qtiles + n_ktiles) > INT_MAX) return FA_ERR_SHAPE;   // one grid
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  if (dv_width != 64 && dv_width != 128) return FA_ERR_UNSUPPORTED_D;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0 || (Nq == 0 && Nk == 0)) return FA_OK;  // nothing to write
  if (Nq > 0 && (!q || !o || !lse || !dout || !dq || !delta)) return FA_ERR_NULLPTR;
  if (Nk > 0 && (!k || !v || !dk || !dv)) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                        reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                        reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv);
  const uintptr_t a4 = reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(delta) |
                       reinterpret_cast<uintptr_t>(seqlens_k);
  if ((a16 & 15u) || (a4 & 3u)) return FA_ERR_ALIGN;
  if (one) {
    // the dQ sum keeps every row of the last tile (the conversion runs one
    // block per (batch*head, query tile), within the grid bound above)
    if (n_qtiles * fa::kBwdTile > INT_MAX) return FA_ERR_SHAPE;
    if (!ws || ws_bytes < static_cast<size_t>(onepass_acc_bytes(bh, Nq, d)))
      return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 15u) return FA_ERR_ALIGN;
  }

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;

  const bool bf16 = dtype == FA_BF16;
  fa::BwdParams p;
  // Without queries or keys no tile of them is ever loaded; the maps still
  // need a row and an address.
  const int nq_rows = Nq > 0 ? Nq : 1, nk_rows = Nk > 0 ? Nk : 1;
  const void* qa = Nq > 0 ? q : k;
  const void* ka = Nk > 0 ? k : q;
  const void* va = Nk > 0 ? v : q;
  const void* da = Nq > 0 ? dout : k;
  if (!make_tmap(&p.tm_q, qa, static_cast<int>(bh), nq_rows, d, bf16) ||
      !make_tmap(&p.tm_k, ka, static_cast<int>(bh), nk_rows, d, bf16) ||
      !make_tmap(&p.tm_v, va, static_cast<int>(bh), nk_rows, dv_width, bf16) ||
      !make_tmap(&p.tm_do, da, static_cast<int>(bh), nq_rows, dv_width, bf16))
    return FA_ERR_TENSORMAP;
  p.width_qk = d;
  p.width_v = dv_width;
  // the kernels are compiled for the larger of the two widths
  const int dk_max = d > dv_width ? d : dv_width;
  p.lse = lse;
  p.delta = delta;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = info->status;
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.N = Nq;
  p.n_tiles = static_cast<int>(n_qtiles);
  p.Nk = Nk;
  p.n_ktiles = static_cast<int>(n_ktiles);
  p.H = H;
  p.seqlens_k = seqlens_k;
  p.align_br = causal == 2 ? 1 : 0;
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.varlen = 0;
  p.total_q = 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  set_dropout(&p, drop_t, seed, drop_off);
  p.dq_acc = static_cast<float*>(ws);
  p.dq_pad = static_cast<int>(n_qtiles * fa::kBwdTile);
  // item order: a head at a time (its tiles share the streamed tiles and,
  // in one pass, the dQ sums in L2) when every tile of a kind costs the
  // same; groups of 8 heads when causal masks or key counts make the
  // tiles' ranges unequal, so the round-robin deal mixes long and short
  p.item_group = (causal || seqlens_k) ? static_cast<int>(bh < 8 ? bh : 8) : 1;
  const bool c = causal != 0;
  cudaError_t e;
  if (one && drop_t < 256)
    e = (d == 64)
            ? fa::launch_bwd_onepass_drop_d64(p, o, dout, delta, bf16, c, info->sms, stream)
            : fa::launch_bwd_onepass_drop_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  else if (one)
    e = (d == 64) ? fa::launch_bwd_onepass_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                  : fa::launch_bwd_onepass_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  else if (kv && drop_t < 256)
    e = (dk_max == 64) ? fa::launch_bwd_kv_drop_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                       : fa::launch_bwd_kv_drop_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  else if (kv)
    e = (dk_max == 64) ? fa::launch_bwd_kv_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                       : fa::launch_bwd_kv_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  else if (drop_t < 256)
    e = (d == 64) ? fa::launch_bwd_drop_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                  : fa::launch_bwd_drop_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  else
    e = (d == 64) ? fa::launch_bwd_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                  : fa::launch_bwd_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H, int N,
           int d, int causal, float scale, int dtype, cudaStream_t stream) {
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, N, d, d, causal, false,
                  nullptr, scale, dtype, 256, 0, 0, stream);
}

int fa_bwd_onepass_workspace_size(int B, int H, int N, int d, size_t* bytes) {
  if (!bytes) return FA_ERR_NULLPTR;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  *bytes = static_cast<size_t>(onepass_acc_bytes(static_cast<long long>(B) * H, N, d));
  return FA_OK;
}

int fa_bwd_onepass(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H,
                   int N, int d, int causal, float scale, int dtype, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, N, d, d, causal, false,
                  nullptr, scale, dtype, 256, 0, 0, stream, true, workspace, workspace_bytes);
}

int fa_bwd_onepass_dropout(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                           float* delta, int B, int H, int N, int d, int causal, float scale,
                           float dropout_p, unsigned long long seed, unsigned int offset,
                           int dtype, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  const int t = drop_threshold(dropout_p);
  if (t < 0) return FA_ERR_DROPOUT;
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, N, d, d, causal, false,
                  nullptr, scale, dtype, t, seed, offset, stream, true, workspace,
                  workspace_bytes);
}

int fa_bwd_kv(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H, int Nq,
              int Nk, int d, int dv_width, int causal, const int* seqlens_k, float scale,
              int dtype, cudaStream_t stream) {
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, d, dv_width, causal,
                  true, seqlens_k, scale, dtype, 256, 0, 0, stream);
}

int fa_bwd_kv_dropout(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      float* delta, int B, int H, int Nq, int Nk, int d, int dv_width, int causal,
                      const int* seqlens_k, float scale, float dropout_p, unsigned long long seed,
                      unsigned int offset, int dtype, cudaStream_t stream) {
  const int t = drop_threshold(dropout_p);
  if (t < 0) return FA_ERR_DROPOUT;
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, d, dv_width, causal,
                  true, seqlens_k, scale, dtype, t, seed, offset, stream);
}

// fa_bwd_varlen, and fa_bwd_varlen_dropout when drop_t < 256.
static int backward_varlen(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                           float* delta, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                           int H, int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                           int d, int dv_width, int causal, float scale, int dtype, int drop_t,
                           unsigned long long seed, unsigned int drop_off, cudaStream_t stream) {
  if (B < 0 || H < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0 ||
      d <= 0 || dv_width <= 0)
    return FA_ERR_SHAPE;
  if (causal < 0 || causal > 2) return FA_ERR_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qtiles = (static_cast<long long>(max_seqlen_q) + fa::kBwdTile - 1) / fa::kBwdTile;
  const long long n_ktiles = (static_cast<long long>(max_seqlen_k) + fa::kBwdTile - 1) / fa::kBwdTile;
  if (bh > INT_MAX || bh * (n_qtiles + n_ktiles) > INT_MAX ||
      static_cast<long long>(total_q) * H > INT_MAX || static_cast<long long>(total_k) * H > INT_MAX)
    return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  if (dv_width != 64 && dv_width != 128) return FA_ERR_UNSUPPORTED_D;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0 || (total_q == 0 && total_k == 0) || (n_qtiles == 0 && n_ktiles == 0)) return FA_OK;
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_NULLPTR;
  if (total_q > 0 && (!q || !o || !lse || !dout || !dq || !delta)) return FA_ERR_NULLPTR;
  if (total_k > 0 && (!k || !v || !dk || !dv)) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                        reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                        reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv);
  const uintptr_t a4 = reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(delta) |
                       reinterpret_cast<uintptr_t>(cu_seqlens_q) |
                       reinterpret_cast<uintptr_t>(cu_seqlens_k);
  if ((a16 & 15u) || (a4 & 3u)) return FA_ERR_ALIGN;

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;

  const bool bf16 = dtype == FA_BF16;
  fa::BwdParams p;
  const int q_tok = total_q > 0 ? total_q : 1, k_tok = total_k > 0 ? total_k : 1;
  const void* qa = total_q > 0 ? q : k;
  const void* da = total_q > 0 ? dout : k;
  const void* ka = total_k > 0 ? k : q;
  const void* va = total_k > 0 ? v : q;
  if (!make_tmap_tokens(&p.tm_q, qa, H, q_tok, d, bf16) ||
      !make_tmap_tokens(&p.tm_k, ka, H, k_tok, d, bf16) ||
      !make_tmap_tokens(&p.tm_v, va, H, k_tok, dv_width, bf16) ||
      !make_tmap_tokens(&p.tm_do, da, H, q_tok, dv_width, bf16))
    return FA_ERR_TENSORMAP;
  p.width_qk = d;
  p.width_v = dv_width;
  const int dk_max = d > dv_width ? d : dv_width;
  p.lse = lse;
  p.delta = delta;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = info->status;
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.N = max_seqlen_q;
  p.n_tiles = static_cast<int>(n_qtiles);
  p.Nk = total_k;
  p.n_ktiles = static_cast<int>(n_ktiles);
  p.H = H;
  p.seqlens_k = nullptr;
  p.align_br = causal == 2 ? 1 : 0;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.varlen = 1;
  p.total_q = total_q;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  set_dropout(&p, drop_t, seed, drop_off);
  p.dq_acc = nullptr;
  p.dq_pad = 0;
  p.item_group = static_cast<int>(bh < 8 ? bh : 8);   // sequences of unequal lengths
  const bool c = causal != 0;
  cudaError_t e;
  if (drop_t < 256)
    e = (dk_max == 64) ? fa::launch_bwd_kv_drop_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                       : fa::launch_bwd_kv_drop_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  else
    e = (dk_max == 64) ? fa::launch_bwd_kv_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                       : fa::launch_bwd_kv_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, float* delta,
                  const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                  int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int d,
                  int dv_width, int causal, float scale, int dtype, cudaStream_t stream) {
  return backward_varlen(q, k, v, o, lse, dout, dq, dk, dv, delta, cu_seqlens_q, cu_seqlens_k, B,
                         H, max_seqlen_q, max_seqlen_k, total_q, total_k, d, dv_width, causal,
                         scale, dtype, 256, 0, 0, stream);
}

int fa_bwd_varlen_dropout(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          float* delta, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                          int H, int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                          int d, int dv_width, int causal, float scale, float dropout_p,
                          unsigned long long seed, unsigned int offset, int dtype,
                          cudaStream_t stream) {
  const int t = drop_threshold(dropout_p);
  if (t < 0) return FA_ERR_DROPOUT;
  return backward_varlen(q, k, v, o, lse, dout, dq, dk, dv, delta, cu_seqlens_q, cu_seqlens_k, B,
                         H, max_seqlen_q, max_seqlen_k, total_q, total_k, d, dv_width, causal,
                         scale, dtype, t, seed, offset, stream);
}

int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H,
                   int N, int d, int causal, float scale, float dropout_p,
                   unsigned long long seed, unsigned int offset, int dtype,
                   cudaStream_t stream) {
  const int t = drop_threshold(dropout_p);
  if (t < 0) return FA_ERR_DROPOUT;
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, N, d, d, causal, false,
                  nullptr, scale, dtype, t, seed, offset, stream);
}

}  // extern "C"

namespace fa {
cudaError_t launch_decode(const DecodeParams& p, void* o, float* lse, int d, bool bf16,
                          cudaStream_t stream);
}

namespace {

// Split of the key axis for fa_decode.  One CTA per SM at a time (its ring
// takes most of the shared memory), so a call takes ceil(CTAs / SMs) waves,
// each as long as a split plus a fixed cost per CTA (query load, pipeline
// fill, partial write; about three tiles' worth).  The plan takes the
// number of splits per head, 1 .. ceil(tiles / 4), that minimises
// waves x (tiles per split + 3) (measured on a 67 MB cache over 8 heads:
// one wave of 19 splits, 39 us, against 47 us for 32 splits in two waves).
struct DecodePlan {
  int splits = 0;
  int tiles_per_split = 0;
  size_t o_bytes = 0;     // partial outputs
  size_t bytes = 0;       // whole workspace (partial outputs, then (m, l) pairs)
};

DecodePlan plan_decode(long long bh, int Nq, int Nk, int d, int sms) {
  DecodePlan dp;
  const int tiles = (Nk + fa::kDecTile - 1) / fa::kDecTile;
  if (tiles == 0 || bh == 0) return dp;
  // Within a number of waves more splits never cost more, so only the
  // largest split count of each wave count (and the cap itself) is tried.
  const long long max_splits = (tiles + 3) / 4;
  long long want = 1, best = -1;
  auto consider = [&](long long sp) {
    if (sp < 1) sp = 1;
    if (sp > max_splits) sp = max_splits;
    const long long per = (tiles + sp - 1) / sp;
    const long long cost = ((bh * sp + sms - 1) / sms) * (per + 3);
    if (best < 0 || cost < best || (cost == best && sp < want)) {
      best = cost;
      want = sp;
    }
  };
  const long long max_waves = (bh * max_splits + sms - 1) / sms;
  for (long long w = 1; w <= max_waves; ++w) consider(w * sms / bh);
  consider(max_splits);
  dp.tiles_per_split = static_cast<int>((tiles + want - 1) / want);
  dp.splits = (tiles + dp.tiles_per_split - 1) / dp.tiles_per_split;
  const size_t parts = static_cast<size_t>(bh) * dp.splits * Nq;
  dp.o_bytes = (parts * d * sizeof(float) + 255) / 256 * 256;
  dp.bytes = dp.o_bytes + (parts * 2 * sizeof(float) + 255) / 256 * 256;
  return dp;
}

int decode_checks(int B, int H, int Nq, int Nk, int d, long long* bh) {
  if (B < 0 || H < 0 || Nk < 0 || d <= 0) return FA_ERR_SHAPE;
  if (Nq < 1 || Nq > fa::kDecMaxQ) return FA_ERR_SHAPE;
  *bh = static_cast<long long>(B) * H;
  if (*bh * Nq > INT_MAX || *bh * ((static_cast<long long>(Nk) + 127) / 128) > INT_MAX)
    return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, size_t* bytes) {
  if (!bytes) return FA_ERR_NULLPTR;
  long long bh = 0;
  const int rc = decode_checks(B, H, Nq, Nk, d, &bh);
  if (rc != FA_OK) return rc;
  *bytes = 0;
  if (bh == 0 || Nk == 0) return FA_OK;
  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  *bytes = plan_decode(bh, Nq, Nk, d, info->sms).bytes;
  return FA_OK;
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, int causal, float scale, int dtype, void* workspace,
              size_t workspace_bytes, cudaStream_t stream) {
  long long bh = 0;
  const int rc = decode_checks(B, H, Nq, Nk, d, &bh);
  if (rc != FA_OK) return rc;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0) return FA_OK;  // nothing to write
  if (!q || !o || !lse || (Nk > 0 && (!k || !v))) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_ALIGN;

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;
  const DecodePlan dp = plan_decode(bh, Nq, Nk, d, info->sms);
  if (dp.bytes > 0) {
    if (!workspace || workspace_bytes < dp.bytes) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGN;
  }
  const bool bf16 = dtype == FA_BF16;
  fa::DecodeParams p;
  if (Nk > 0 && (!make_tmap(&p.tm_k, k, static_cast<int>(bh), Nk, d, bf16) ||
                 !make_tmap(&p.tm_v, v, static_cast<int>(bh), Nk, d, bf16)))
    return FA_ERR_TENSORMAP;
  p.q = q;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = dp.bytes ? reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + dp.o_bytes)
                       : nullptr;
  p.status = info->status;
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.Nq = Nq;
  p.Nk = Nk;
  p.splits = dp.splits;
  p.tiles_per_split = dp.tiles_per_split;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  const cudaError_t e = fa::launch_decode(p, o, lse, d, bf16, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // extern "C"
