// Host-buffer executor: C = A·B in FP32 for A, B and C in host memory.
//
// The pages time the kernel on device buffers; a caller whose operands live
// in host memory also pays for moving 2(MK + KN) + 4MN bytes over the
// CPU-GPU link, at about a tenth of HBM bandwidth on GB300.  This executor
// hides most of that behind the GEMM itself, with three streams of its own
// per device (copies in, GEMMs, copies out) ordered by events:
//
//  * K steps.  When K is long enough, B's rows and A's columns cross the
//    link in K blocks, a short first block so that the first GEMM can start
//    early.  Each step computes C over all M rows for its block as soon as
//    the block has landed, continuing every element's FMA chain from the
//    previous step's C (GEMM_OPT_ACCUMULATE), so the result is the one-call
//    FMA chain, bit for bit.
//  * Row chunks.  The last step (or the only one, for short K) runs in row
//    chunks, each copied out as soon as its GEMM is done, the last chunk
//    about one wave of tiles so that little remains to copy once the GPU is
//    done.  With a single step, A crosses the link chunk by chunk as well.
//
// Every copy is one cudaMemcpy2DAsync (a row-pitched block), every GEMM one
// gemm_f32_ws call.  Calls are serialised per device: the streams, events
// and (when the caller reuses it) the scratch space are shared, so each call
// starts after the previous one on the device has finished.
#include <atomic>
#include <mutex>

#include "f32_schedule.cuh"
#include "gemm_internal.h"
#include "pipelined_gemm_testing.h"

namespace pg {

namespace {

constexpr int kMaxKBlocks = 16;
constexpr int kMaxRowChunks = 64;
constexpr int kMaxCompStreams = 3;
constexpr int kEvents = 256;

// Schedule policy.  Measured on GB300 at 4096^3 with pinned host buffers
// (link: about 208 GB/s to the device, 191 GB/s back), TMA fill, two
// stages, ms per call: K blocks 512 / 1280 / 1280 / 1024 with row chunks
// of three and one waves 2.72; 512 / 2048 / 1536 2.64; 512 / 1536 / 2048
// with chunks of two and one waves 2.63; one block 2.88; first blocks of
// 256 or 1024, middle blocks of at most 1024 or 3072, two or three GEMM
// streams, chunk GEMMs without the K split: all slower.  The last block
// runs as row chunks so that copying C out overlaps its GEMMs; what stays
// exposed is the first block's copy in (16 MB), the last chunk's copy out
// and the K steps' shorter, less efficient GEMMs (2.45 ms of GEMMs against
// 2.27 for one call).
struct HostPolicy {
    int k_first = 512;       // first K block: 2 x 8 MB to land before the first GEMM
    int k_last = 2048;       // last K block, run in row chunks
    int k_mid_max = 2048;    // longest block between them
    int k_steps_min = 2048;  // shorter K runs as one step
    int last_rows_waves100 = 100; // last row chunk: about one wave of 128 x 128 tiles
    int rows_waves100 = 200;      // other row chunks: about two waves
    int comp_streams = 1;         // GEMM streams; with more than one, every step runs per row chunk
    int split = 1;                // K-split of the last round of tiles (hand-over workspace)
    int round_chunks = 1;         // first row chunks a whole number of rounds of tiles on the SMs
};

std::atomic<int> g_policy[6] = {{0}, {0}, {0}, {0}, {0}, {0}}; // test overrides, 0: default
std::atomic<int> g_comp_streams{0};                                // test override, 0: default
std::atomic<int> g_split{-1};                                      // test override, -1: default
std::atomic<int> g_round_chunks{-1};                               // test override, -1: default

HostPolicy policy()
{
    HostPolicy p;
    int *fields[6] = {&p.k_first, &p.k_last, &p.k_mid_max, &p.k_steps_min, &p.last_rows_waves100, &p.rows_waves100};
    for (int i = 0; i < 6; ++i) {
        const int v = g_policy[i].load();
        if (v > 0)
            *fields[i] = v;
    }
    if (g_comp_streams.load() > 0)
        p.comp_streams = g_comp_streams.load();
    if (g_split.load() >= 0)
        p.split = g_split.load();
    if (g_round_chunks.load() >= 0)
        p.round_chunks = g_round_chunks.load();
    return p;
}

int round_up(long long x, int m) { return static_cast<int>((x + m - 1) / m * m); }

struct HostSchedule {
    int n_k = 0;
    int k[kMaxKBlocks + 1];
    int n_r = 0;
    int r[kMaxRowChunks + 1];
};

HostSchedule make_schedule(int M, int N, int K, int sms, const HostPolicy &pol)
{
    HostSchedule s;
    // K blocks: [0, first), middle blocks of at most k_mid_max, then the
    // last block from a multiple of 16 at or below K - last.  Every bound but
    // K is a multiple of 16 floats, so every block of A starts on a 64-byte
    // boundary of its row.
    const int first = round_up(pol.k_first, 16);
    const int last = round_up(pol.k_last, 16);
    int n = 0;
    s.k[n++] = 0;
    if (K >= pol.k_steps_min && K >= first + last + 16) {
        const int last_start = (K - last) / 16 * 16;
        if (last_start - first < first / 2) { // no room for a middle block: two blocks
            s.k[n++] = last_start;
            s.k[n++] = K;
            s.n_k = n - 1;
            goto rows;
        }
        s.k[n++] = first;
        const int mid = last_start - first;
        int parts = (mid + pol.k_mid_max - 1) / pol.k_mid_max;
        if (parts > kMaxKBlocks - 2)
            parts = kMaxKBlocks - 2;
        if (parts < 1)
            parts = 1;
        const int step = round_up((mid + parts - 1) / parts, 16);
        for (int b = first + step; b < last_start; b += step)
            s.k[n++] = b;
        if (last_start > first)
            s.k[n++] = last_start;
    }
    s.k[n++] = K;
    s.n_k = n - 1;

rows:
    // Row chunks of the last step: about rows_waves of tiles each, then a
    // last chunk of about last_rows_waves.
    const long long tiles_n = N > 0 ? (N + 127) / 128 : 1;
    const long long wave_rows = (sms + tiles_n - 1) / tiles_n * 128;
    long long last_rows = round_up(wave_rows * pol.last_rows_waves100 / 100, 128);
    long long big_rows = round_up(wave_rows * pol.rows_waves100 / 100, 128);
    if (last_rows < 128)
        last_rows = 128;
    if (big_rows < 128)
        big_rows = 128;
    s.r[0] = 0;
    s.n_r = 0;
    if (M <= last_rows) {
        s.r[++s.n_r] = M;
        return s;
    }
    const long long rest = (M - last_rows) / 128 * 128; // the last chunk takes the ragged rows
    if (rest == 0) {
        s.r[++s.n_r] = M;
        return s;
    }
    // A chunk whose tiles fill whole rounds of SMs runs in the one-tile
    // kernel alone, faster than the split schedule's persistent kernel: with
    // round_chunks the first chunk is the largest such block of rows of at
    // most two usual chunks, if there is one.
    long long start = 0;
    if (pol.round_chunks) {
        long long g = sms, t = tiles_n; // gcd
        while (t != 0) {
            const long long r = g % t;
            g = t;
            t = r;
        }
        const long long unit = sms / g * 128; // rows of a whole number of rounds
        // at most two usual chunks' worth, so that its copy out still
        // overlaps the GEMMs of the chunks after it
        const long long cap = rest < 2 * big_rows ? rest : 2 * big_rows;
        const long long fit = cap / unit * unit;
        if (fit >= unit && fit >= big_rows && fit < rest) {
            s.r[++s.n_r] = static_cast<int>(fit);
            start = fit;
        }
    }
    if (start == rest) {
        s.r[++s.n_r] = M;
        return s;
    }
    // The rows between: `parts` chunks of whole 128-row tiles, as equal as
    // the tile rows allow.
    long long parts = (rest - start + big_rows - 1) / big_rows;
    if (parts > kMaxRowChunks - 2)
        parts = kMaxRowChunks - 2;
    const long long tile_rows = (rest - start) / 128;
    long long b = start;
    for (long long i = 0; i < parts; ++i) {
        b += (tile_rows / parts + (i < tile_rows % parts ? 1 : 0)) * 128;
        s.r[++s.n_r] = static_cast<int>(b);
    }
    s.r[++s.n_r] = M;
    return s;
}

// Streams and events of one device context, made on first use.
struct HostHandles {
    unsigned long long ctx = 0;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaStream_t comp[kMaxCompStreams] = {};
    cudaEvent_t ev[kEvents] = {};
    cudaEvent_t prev_end = nullptr; // end of the previous call on this device
    bool prev_valid = false;
};

struct HostResources {
    std::mutex lock;
    HostHandles h;
};

HostResources g_res[kMaxDevices];

int ensure_handles(HostHandles &h, unsigned long long ctx)
{
    if (h.h2d != nullptr && h.ctx == ctx)
        return GEMM_OK;
    // A new context: the old handles belonged to one that is gone (after
    // cudaDeviceReset), so they are dropped rather than destroyed.
    h = HostHandles{};
    bool made = cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking) == cudaSuccess;
    for (auto &c : h.comp)
        made = made && cudaStreamCreateWithFlags(&c, cudaStreamNonBlocking) == cudaSuccess;
    if (!made) {
        h = HostHandles{};
        return GEMM_ERR_CUDA;
    }
    for (auto &e : h.ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            h = HostHandles{};
            return GEMM_ERR_CUDA;
        }
    if (cudaEventCreateWithFlags(&h.prev_end, cudaEventDisableTiming) != cudaSuccess) {
        h = HostHandles{};
        return GEMM_ERR_CUDA;
    }
    h.ctx = ctx;
    return GEMM_OK;
}

constexpr size_t kScratchAlign = 256;

size_t align_up(size_t x) { return (x + kScratchAlign - 1) / kScratchAlign * kScratchAlign; }

struct ScratchLayout {
    int lda, ldb, ldc; // device leading dimensions: 16-byte row pitches
    size_t a, b, c, ws, ws_bytes, total; // ws: kMaxCompStreams hand-over spaces of ws_bytes each
};

ScratchLayout scratch_layout(int M, int N, int K, int sms)
{
    ScratchLayout l;
    l.lda = round_up(K > 0 ? K : 1, 4);
    l.ldb = round_up(N > 0 ? N : 1, 4);
    l.ldc = l.ldb;
    l.a = 0;
    l.b = align_up(l.a + static_cast<size_t>(M) * l.lda * 4);
    l.c = align_up(l.b + static_cast<size_t>(K) * l.ldb * 4);
    l.ws = align_up(l.c + static_cast<size_t>(M) * l.ldc * 4);
    l.ws_bytes = static_cast<size_t>(f32_handover_bytes(sms));
    l.total = l.ws + kMaxCompStreams * align_up(l.ws_bytes);
    return l;
}

} // namespace

} // namespace pg

using namespace pg;

extern "C" int gemm_f32_host_scratch(int M, int N, int K, size_t *bytes)
{
    if (M < 0 || N < 0 || K < 0 || bytes == nullptr)
        return GEMM_ERR_INVALID_ARG;
    *bytes = scratch_layout(M, N, K, device_sms()).total;
    return GEMM_OK;
}

extern "C" int gemm_f32_host_schedule(int M, int N, int K, int sms, int *k_bounds, int k_cap, int *n_k,
                                      int *row_bounds, int row_cap, int *n_rows)
{
    if (M < 0 || N < 0 || K < 0 || sms < 1 || !k_bounds || !n_k || !row_bounds || !n_rows)
        return GEMM_ERR_INVALID_ARG;
    const HostSchedule s = make_schedule(M, N, K, sms, policy());
    if (k_cap < s.n_k + 1 || row_cap < s.n_r + 1)
        return GEMM_ERR_INVALID_ARG;
    for (int i = 0; i <= s.n_k; ++i)
        k_bounds[i] = s.k[i];
    for (int i = 0; i <= s.n_r; ++i)
        row_bounds[i] = s.r[i];
    *n_k = s.n_k;
    *n_rows = s.n_r;
    return GEMM_OK;
}

extern "C" int gemm_testing_host_policy(int k_first, int k_last, int k_mid_max, int k_steps_min,
                                        int last_rows_waves100, int rows_waves100)
{
    const int v[6] = {k_first, k_last, k_mid_max, k_steps_min, last_rows_waves100, rows_waves100};
    for (int x : v)
        if (x < 0)
            return GEMM_ERR_INVALID_ARG;
    if ((k_first > 0 && k_first < 16) || (k_last > 0 && k_last < 16) || (k_mid_max > 0 && k_mid_max < 16))
        return GEMM_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        g_policy[i].store(v[i]);
    return GEMM_OK;
}

extern "C" int gemm_testing_host_streams(int comp_streams, int split, int round_chunks)
{
    if (comp_streams < 0 || comp_streams > kMaxCompStreams || split < -1 || split > 1 || round_chunks < -1 ||
        round_chunks > 1)
        return GEMM_ERR_INVALID_ARG;
    g_comp_streams.store(comp_streams);
    g_split.store(split);
    g_round_chunks.store(round_chunks);
    return GEMM_OK;
}

extern "C" int gemm_f32_host(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C,
                             int ldc, int fill_mode, int stages, int block_tile, void *scratch,
                             size_t scratch_bytes, unsigned int *status_out, void *stream)
{
    if ((fill_mode & GEMM_OPT_ACCUMULATE) != 0)
        return GEMM_ERR_INVALID_ARG; // this entry computes C = A·B; it uses the option itself
    // Host operands: any row pitch at least their width, 4-byte aligned.
    if (M < 0 || N < 0 || K < 0 || lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
        return GEMM_ERR_INVALID_ARG;
    if (M > 0 && N > 0 && (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))))
        return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 3u)
        return GEMM_ERR_MISALIGNED;
    // The GEMMs run on the device copies, whose rows start on 16-byte
    // boundaries: the whole problem's plan in that layout validates the fill,
    // stages, tile and options, and decides the tile every call uses.
    const ScratchLayout L0 = scratch_layout(M, N, K, 1);
    const float *dev_base = reinterpret_cast<const float *>(static_cast<uintptr_t>(kScratchAlign));
    gemm_plan plan;
    int st = gemm_f32_plan(M, N, K, dev_base, L0.lda, dev_base, L0.ldb, const_cast<float *>(dev_base), L0.ldc,
                           fill_mode, stages, block_tile, &plan);
    if (st != GEMM_OK)
        return st;
    if (status_out)
        *status_out = 0;
    if (M == 0 || N == 0)
        return GEMM_OK;
    int dev;
    st = device_checked(&dev);
    if (st != GEMM_OK)
        return st;
    const int sms = device_sms();
    const ScratchLayout L = scratch_layout(M, N, K, sms);
    if (scratch == nullptr || scratch_bytes < L.total)
        return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(scratch) & (kScratchAlign - 1)) != 0)
        return GEMM_ERR_MISALIGNED;
    const HostPolicy P = policy();
    const HostSchedule S = make_schedule(M, N, K, sms, P);
    const int nc = P.comp_streams < 1 ? 1 : P.comp_streams > kMaxCompStreams ? kMaxCompStreams : P.comp_streams;
    const unsigned long long ctx = current_context_id();

    HostResources &R = g_res[dev];
    std::lock_guard<std::mutex> guard(R.lock);
    st = ensure_handles(R.h, ctx);
    if (st != GEMM_OK)
        return st;
    HostHandles &H = R.h;

    uint8_t *base = static_cast<uint8_t *>(scratch);
    float *Ad = reinterpret_cast<float *>(base + L.a);
    float *Bd = reinterpret_cast<float *>(base + L.b);
    float *Cd = reinterpret_cast<float *>(base + L.c);
    // One hand-over space per GEMM stream: calls on one stream never
    // overlap, calls on two may.
    auto ws_of = [&](cudaStream_t cs) -> void * {
        for (int c = 0; c < nc; ++c)
            if (H.comp[c] == cs)
                return base + L.ws + c * align_up(L.ws_bytes);
        return nullptr;
    };
    const int tile = plan.block_m;
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    int evi = 0;
    const size_t fsz = sizeof(float);

    auto copy_a = [&](int r0, int r1, int k0, int k1) {
        return cudaMemcpy2DAsync(Ad + static_cast<size_t>(r0) * L.lda + k0, L.lda * fsz,
                                 A + static_cast<size_t>(r0) * lda + k0, static_cast<size_t>(lda) * fsz,
                                 static_cast<size_t>(k1 - k0) * fsz, static_cast<size_t>(r1 - r0),
                                 cudaMemcpyHostToDevice, H.h2d) == cudaSuccess;
    };
    auto copy_b = [&](int k0, int k1) {
        return cudaMemcpy2DAsync(Bd + static_cast<size_t>(k0) * L.ldb, L.ldb * fsz,
                                 B + static_cast<size_t>(k0) * ldb, static_cast<size_t>(ldb) * fsz,
                                 static_cast<size_t>(N) * fsz, static_cast<size_t>(k1 - k0),
                                 cudaMemcpyHostToDevice, H.h2d) == cudaSuccess;
    };
    auto copy_c = [&](int r0, int r1) {
        return cudaMemcpy2DAsync(C + static_cast<size_t>(r0) * ldc, static_cast<size_t>(ldc) * fsz,
                                 Cd + static_cast<size_t>(r0) * L.ldc, L.ldc * fsz, static_cast<size_t>(N) * fsz,
                                 static_cast<size_t>(r1 - r0), cudaMemcpyDeviceToHost, H.d2h) == cudaSuccess;
    };
    // `to` waits for everything issued to `from` so far.
    auto join = [&](cudaStream_t from, cudaStream_t to) {
        if (evi >= kEvents)
            return false;
        cudaEvent_t e = H.ev[evi++];
        return cudaEventRecord(e, from) == cudaSuccess && cudaStreamWaitEvent(to, e, 0) == cudaSuccess;
    };
    auto gemm = [&](cudaStream_t cs, int r0, int r1, int k0, int k1, bool accumulate) {
        return gemm_f32_ws(r1 - r0, N, k1 - k0, Ad + static_cast<size_t>(r0) * L.lda + k0, L.lda,
                           Bd + static_cast<size_t>(k0) * L.ldb, L.ldb, Cd + static_cast<size_t>(r0) * L.ldc, L.ldc,
                           fill_mode | (accumulate ? GEMM_OPT_ACCUMULATE : 0), stages, tile,
                           P.split ? ws_of(cs) : nullptr, P.split ? L.ws_bytes : 0, cs);
    };
    // Row chunk i's GEMMs run on comp[i % nc]: its C rows are only ever
    // touched by that stream.
    auto comp_of = [&](int i) { return H.comp[i % nc]; };

    // Start after the caller's stream and after the previous call on this
    // device, which may still be using a scratch space the caller reuses.
    bool ok = join(user, H.h2d) && join(user, H.d2h);
    for (int c = 0; c < nc; ++c)
        ok = ok && join(user, H.comp[c]);
    if (ok && H.prev_valid) {
        ok = cudaStreamWaitEvent(H.h2d, H.prev_end, 0) == cudaSuccess &&
             cudaStreamWaitEvent(H.d2h, H.prev_end, 0) == cudaSuccess;
        for (int c = 0; c < nc; ++c)
            ok = ok && cudaStreamWaitEvent(H.comp[c], H.prev_end, 0) == cudaSuccess;
    }
    st = ok ? GEMM_OK : GEMM_ERR_CUDA;
    // h2d's progress so far, made visible to every GEMM stream.
    auto publish_h2d = [&]() {
        if (evi >= kEvents)
            return false;
        cudaEvent_t e = H.ev[evi++];
        if (cudaEventRecord(e, H.h2d) != cudaSuccess)
            return false;
        for (int c = 0; c < nc; ++c)
            if (cudaStreamWaitEvent(H.comp[c], e, 0) != cudaSuccess)
                return false;
        return true;
    };
    if (st == GEMM_OK && S.n_k == 1) {
        // One step: all of B, then A, the GEMM and C chunk by chunk (K = 0:
        // nothing to copy in; the GEMMs write the empty sum's zeros).
        if (K > 0 && !copy_b(0, K))
            st = GEMM_ERR_CUDA;
        for (int i = 0; st == GEMM_OK && i < S.n_r; ++i) {
            const int r0 = S.r[i], r1 = S.r[i + 1];
            cudaStream_t cs = comp_of(i);
            if ((K > 0 && !copy_a(r0, r1, 0, K)) || !join(H.h2d, cs))
                st = GEMM_ERR_CUDA;
            else if ((st = gemm(cs, r0, r1, 0, K, false)) == GEMM_OK && (!join(cs, H.d2h) || !copy_c(r0, r1)))
                st = GEMM_ERR_CUDA;
        }
    } else if (st == GEMM_OK) {
        // K steps, the last one (or, with several GEMM streams, every one)
        // in row chunks.
        for (int j = 0; st == GEMM_OK && j < S.n_k; ++j) {
            const int k0 = S.k[j], k1 = S.k[j + 1];
            const bool last = j + 1 == S.n_k;
            if (!copy_a(0, M, k0, k1) || !copy_b(k0, k1) || !publish_h2d()) {
                st = GEMM_ERR_CUDA;
                break;
            }
            if (!last && nc == 1) {
                st = gemm(H.comp[0], 0, M, k0, k1, j > 0);
                continue;
            }
            for (int i = 0; st == GEMM_OK && i < S.n_r; ++i) {
                const int r0 = S.r[i], r1 = S.r[i + 1];
                cudaStream_t cs = comp_of(i);
                if ((st = gemm(cs, r0, r1, k0, k1, j > 0)) == GEMM_OK && last &&
                    (!join(cs, H.d2h) || !copy_c(r0, r1)))
                    st = GEMM_ERR_CUDA;
            }
        }
    }
    // Whatever was issued, d2h ends after all of it; the caller's stream and
    // the next call wait for that point.  (On success the last copy out
    // already follows every GEMM, and every GEMM every copy in.)
    evi = evi > kEvents - 1 - nc ? kEvents - 1 - nc : evi;
    bool joined = join(H.h2d, H.d2h);
    for (int c = 0; c < nc; ++c)
        joined = joined && join(H.comp[c], H.d2h);
    // The status word, read and cleared after the last GEMM, as
    // gemm_device_status does, without a synchronisation of its own.
    if (joined && status_out) {
        unsigned int *word = device_status_word(dev, ctx);
        joined = word != nullptr &&
                 cudaMemcpyAsync(status_out, word, sizeof *word, cudaMemcpyDeviceToHost, H.d2h) == cudaSuccess &&
                 cudaMemsetAsync(word, 0, sizeof *word, H.d2h) == cudaSuccess;
    }
    joined = joined && cudaEventRecord(H.prev_end, H.d2h) == cudaSuccess &&
             cudaStreamWaitEvent(user, H.prev_end, 0) == cudaSuccess;
    H.prev_valid = joined;
    if (!joined && st == GEMM_OK)
        st = GEMM_ERR_CUDA;
    return st;
}
