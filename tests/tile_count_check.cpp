// Host check of the tile walk of the ring kernels: for every layout, mask,
// ring size, chunk length (tile-aligned or ragged) and tile width, and every
// last query slot a rank can hold, the whole-ring tile count (closed form)
// equals the sum of the per-step counts and the number of tiles the walk
// itself visits.  Prints one line per failure and exits 1 if any.
#include <cstdio>

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
    std::printf("%ld (geometry, tile, last query) cases, %d mismatches\n", cases, bad);
    return bad ? 1 : 0;
}
