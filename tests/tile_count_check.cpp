// Host check of the tile walk of the ring kernels: for every layout, mask,
// ring size, chunk length (tile-aligned or ragged) and tile width, and every
// last query slot a rank can hold, the whole-ring tile count (closed form)
// equals the sum of the per-step counts and the number of tiles the walk
// itself visits.  Also: both unit numberings (heads fastest, and each
// (batch, head) contiguous) reach every (batch, head, query tile) of the
// selected ranks exactly once.  Prints one line per failure and exits 1 if any.
#include <cstdio>
#include <set>
#include <tuple>

#include "cp_common.cuh"

using namespace cp;

template <int T>
static int check(const Geom &g)
{
    int bad = 0;
    for (int r = 0; r < g.N; ++r)
        for (int i = 0; i < g.cpr; ++i) {
            const int ch = rank_chunk(g, r, i);
            for (int u = ch * g.clen; u < (ch + 1) * g.clen; ++u) {
                const int closed = KvIter<T>::count(g, r, u);
                int steps = 0;
                for (int k = 0; k < g.N; ++k) steps += KvIter<T>::count(g, r, u, k, k + 1);
                int walked = 0;
                KvIter<T> it;
                for (it.begin(g, r, u); it.valid(); it.next()) ++walked;
                if (closed != steps || closed != walked) {
                    if (++bad <= 5)
                        std::printf("T=%d S=%d N=%d layout=%d causal=%d r=%d qmax=%d: closed %d, steps %d, walk %d\n",
                                    T, g.S, g.N, g.layout, g.causal, r, u, closed, steps, walked);
                }
            }
        }
    return bad;
}

static int check_units(const Geom &g, int B, int Hq, int lo, int hi, bool grouped)
{
    const int qrows = 128, upc = (g.clen + qrows - 1) / qrows;
    const int units = num_selected_chunks(g, lo, hi) * upc * B * Hq;
    std::set<std::tuple<int, int, int>> seen;   // (b, h, q0)
    int bad = 0;
    for (int u = 0; u < units; ++u) {
        const Unit w = grouped ? decode_unit_grouped(g, B, Hq, upc, qrows, u)
                               : decode_unit(g, B, Hq, lo, hi, upc, qrows, u);
        const int ch = w.q0 / g.clen;
        const bool held = w.r >= lo && w.r < hi && chunk_rank(g, ch) == w.r && w.q0 >= ch * g.clen &&
                          w.qmax < (ch + 1) * g.clen && w.qmax >= w.q0 && (w.q0 - ch * g.clen) % qrows == 0;
        if (!held || w.b < 0 || w.b >= B || w.h < 0 || w.h >= Hq || !seen.insert({w.b, w.h, w.q0}).second) ++bad;
    }
    if (bad)
        std::printf("units S=%d N=%d layout=%d B=%d Hq=%d ranks [%d,%d) grouped=%d: %d bad\n", g.S, g.N, g.layout,
                    B, Hq, lo, hi, (int)grouped, bad);
    return bad;
}

int main()
{
    const int Ns[] = {1, 2, 3, 4, 8, 16};
    const int clens[] = {1, 7, 64, 127, 128, 129, 255, 256, 257, 300, 512, 1000};
    long cases = 0;
    int bad = 0;
    for (int layout = 0; layout < 3; ++layout)
        for (int causal = 0; causal < 2; ++causal)
            for (int N : Ns)
                for (int clen : clens) {
                    const int cpr = layout == CP_LAYOUT_ZIGZAG ? 2 : 1;
                    const Geom g = make_geom(N * cpr * clen, N, layout, causal);
                    bad += check<64>(g) + check<128>(g) + check<256>(g);
                    cases += 3L * g.S;
                }
    for (int layout = 0; layout < 3; ++layout)
        for (int N : {1, 2, 4, 8})
            for (int clen : {128, 300, 1024}) {
                const int cpr = layout == CP_LAYOUT_ZIGZAG ? 2 : 1;
                const Geom g = make_geom(N * cpr * clen, N, layout, 1);
                bad += check_units(g, 2, 3, 0, N, false) + check_units(g, 2, 3, 0, N, true) +
                       check_units(g, 1, 2, N / 2, N, false);
            }
    std::printf("%ld (geometry, tile, last query) cases, %d mismatches\n", cases, bad);
    return bad ? 1 : 0;
}
