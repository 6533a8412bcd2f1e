// Work schedule of the persistent FP32 TMA kernel: which (tile, K-slice
// range) pieces each CTA computes, and in what order.  Plain integer
// arithmetic, usable on the host (planning, tests) and on the device.
//
// P persistent CTAs walk the T tiles in rounds (tile r*P + c for CTA c).
// When T is not a multiple of P, the last round would leave SMs idle, so the
// last P + (T mod P) tiles form a split region instead: its
// (P + T mod P) * k slice-units (k slices per tile, tile-major) are dealt to
// the CTAs in equal contiguous ranges, each at least one tile long.  A tile
// cut by a range boundary is computed in two pieces, in K order: the CTA
// whose range ends inside it computes slices [0, s) (the head) and hands its
// FP32 accumulators to the next CTA, which computes slices [s, k) (the tail)
// starting from them.  Every C element is therefore still one FMA chain over
// k ascending from +0, exactly as in an unsplit tile: the split moves work,
// not arithmetic.
//
// Order within a CTA: whole-tile rounds, then its head piece (if any), then
// the whole tiles of its range, then its tail piece (if any).  A CTA's head
// is the first thing it does in the region and a tail the last, and every
// range is at least one tile long, so a tail's head has normally been
// finished long before it is needed (the head took at most one tile's
// slices; the tail starts after at least that many).
#pragma once

namespace pg {

struct F32Piece {
    int tile;          // linear tile index
    int s_begin;       // first K slice
    int s_end;         // one past the last K slice
    bool from_partial; // starts from the accumulators the previous CTA handed over
    bool to_partial;   // hands its accumulators to the next CTA instead of writing C
};

struct F32Schedule {
    int tiles;          // T
    int ctas;           // P
    int k;              // K slices per tile
    int whole_rounds;   // rounds of whole tiles before the split region
    int region0;        // first tile of the split region
    long long units;    // slice-units of the split region (0: no split)

    __host__ __device__ static F32Schedule make(int tiles, int ctas, int k, bool allow_split)
    {
        F32Schedule s;
        s.tiles = tiles;
        s.ctas = ctas;
        s.k = k;
        const int rounds = ctas > 0 ? tiles / ctas : 0;
        const int rem = ctas > 0 ? tiles % ctas : 0;
        if (allow_split && rounds >= 1 && rem != 0 && k >= 2) {
            s.whole_rounds = rounds - 1;
            s.region0 = s.whole_rounds * ctas;
            s.units = static_cast<long long>(tiles - s.region0) * k;
        } else {
            s.whole_rounds = ctas > 0 ? (tiles + ctas - 1) / ctas : 0;
            s.region0 = tiles;
            s.units = 0;
        }
        return s;
    }

    __host__ __device__ bool split() const { return units != 0; }
};

// The pieces of one CTA, worked out once: CTA c's range of the split region
// is slice-units [units * c / P, units * (c + 1) / P), so it begins with the
// tail of a tile the CTA before it started (unless the range starts on a tile
// boundary), covers some whole tiles, and ends with the head of a tile the
// next CTA finishes (unless it ends on a boundary).  The 64-bit divisions
// happen here, once; walking the pieces then takes a few 32-bit comparisons
// (a persistent kernel's K loop ran several per cent slower with the
// divisions at every piece).
struct F32CtaPieces {
    int ctas, cta, k;
    int whole;      // whole-tile rounds: tiles cta, cta + ctas, ...
    int head_tile;  // tile whose first head_end slices this CTA hands over (-1: none)
    int head_end;
    int full_first; // whole tiles of the split region: [full_first, full_first + full_count)
    int full_count;
    int tail_tile;  // tile this CTA finishes from slice tail_begin (-1: none)
    int tail_begin;

    __host__ __device__ static F32CtaPieces make(const F32Schedule &s, int c)
    {
        F32CtaPieces q;
        q.ctas = s.ctas;
        q.cta = c;
        q.k = s.k;
        q.whole = 0;
        if (!s.split()) {
            // whole rounds while tile r * ctas + c exists
            q.whole = c < s.tiles ? (s.tiles - 1 - c) / s.ctas + 1 : 0;
        } else {
            q.whole = s.whole_rounds;
        }
        q.head_tile = q.tail_tile = -1;
        q.head_end = q.tail_begin = 0;
        q.full_first = q.full_count = 0;
        if (s.split()) {
            const long long u0 = s.units * c / s.ctas;
            const long long u1 = s.units * (c + 1) / s.ctas;
            if (u1 % s.k != 0) {
                q.head_tile = s.region0 + static_cast<int>(u1 / s.k);
                q.head_end = static_cast<int>(u1 % s.k);
            }
            const long long first_full = (u0 + s.k - 1) / s.k;
            q.full_first = s.region0 + static_cast<int>(first_full);
            q.full_count = static_cast<int>(u1 / s.k - first_full);
            if (u0 % s.k != 0) {
                q.tail_tile = s.region0 + static_cast<int>(u0 / s.k);
                q.tail_begin = static_cast<int>(u0 % s.k);
            }
        }
        return q;
    }

    __host__ __device__ int count() const
    {
        return whole + (head_tile >= 0 ? 1 : 0) + full_count + (tail_tile >= 0 ? 1 : 0);
    }

    // Piece idx, 0 <= idx < count(): whole rounds, the head, the region's
    // whole tiles, the tail.
    __host__ __device__ F32Piece piece(int idx) const
    {
        if (idx < whole)
            return F32Piece{idx * ctas + cta, 0, k, false, false};
        idx -= whole;
        if (head_tile >= 0) {
            if (idx == 0)
                return F32Piece{head_tile, 0, head_end, false, true};
            --idx;
        }
        if (idx < full_count)
            return F32Piece{full_first + idx, 0, k, false, false};
        return F32Piece{tail_tile, tail_begin, k, true, false};
    }
};

// Bytes of hand-over space a split schedule over `ctas` CTAs needs: one
// 128 x 128 FP32 accumulator tile per CTA (a CTA hands over at most one) and
// one 8-byte ready flag per CTA.
constexpr long long kF32HandoverTileBytes = 128LL * 128 * 4;

__host__ __device__ inline long long f32_handover_bytes(int ctas)
{
    return static_cast<long long>(ctas) * (kF32HandoverTileBytes + 8);
}

} // namespace pg
