// Host-side check of the decode kernels' work schedule (the quota rule and the piece
// cursor of decode_tc.cuh, compiled for the host). Reads cases from stdin, one per line:
//     B S pairs L_0 ... L_{B-1}
// and for each prints "ok <max tiles of a pair> <ceil(T / pairs)> <pieces> <split>" or
// "fail <reason>" (split: the pieces per sequence of the split plan, 0 for the tile plan).
// Every pair's share is set up the way the kernel's sched_init does it (tile counts,
// their prefix sums and sched_plan), then walked piece by piece.
#include <cstdio>
#include <cstdlib>
#include <string>
#include <vector>

#include "decode_tc.cuh"

using namespace mla;

static std::string run_case(int B, int S, int pairs, const std::vector<int32_t>& lens, long long* max_tiles,
                            long long* ideal, long long* npieces, int* split) {
  DecodeParams p{};
  p.B = B;
  p.S = S;
  p.S_used = S;
  p.balanced = 1;
  p.pairs = pairs;
  p.n_h = 128;
  p.seq_lens = lens.data();
  std::vector<long long> tiles(B), first(B);
  long long T = 0;
  int Tmax = 0;
  for (int b = 0; b < B; ++b) {
    tiles[b] = (std::max(lens[b], 0) + kSchedTile - 1) / kSchedTile;
    first[b] = T;
    T += tiles[b];
    Tmax = std::max<int>(Tmax, (int)tiles[b]);
  }
  int Tmin = B > 0 ? (int)tiles[0] : 0;
  for (int b = 0; b < B; ++b) Tmin = std::min<int>(Tmin, (int)tiles[b]);
  *ideal = (T + pairs - 1) / pairs;
  *max_tiles = 0;
  *npieces = 0;
  std::vector<std::vector<char>> covered(B);
  for (int b = 0; b < B; ++b) covered[b].assign(std::max(lens[b], 0), 0);
  std::vector<int> next_slot(B, 0), lasts(B, 0);
  long long quota = 0;
  for (int pr = 0; pr < pairs; ++pr) {
    SchedShared sh{};
    int bn = 0;
    int64_t bc = -1;
    if (Tmin == Tmax && Tmax >= 1) sched_best_split(B, Tmax, S, pairs, &bn, &bc);
    sched_plan(T, B, Tmin, Tmax, S, pairs, pr, bn, bc, &sh);
    *split = sh.split;
    if (sh.split > 0) {
      quota = (((long long)B * sh.split + pairs - 1) / pairs) * sh.per;
    } else {
      quota = sh.q;
    }
    sh.b0 = -1;
    for (int b = 0; b < B && sh.split == 0 && sh.t_begin < sh.t_end; ++b)
      if (first[b] <= sh.t_begin && sh.t_begin < first[b] + tiles[b]) {
        sh.b0 = b;
        sh.c0 = first[b];
        break;
      }
    PieceCursor cur;
    cur.start(p, pr, sh);
    Piece pc;
    long long mine = 0;
    while (cur.next(p, pc)) {
      ++*npieces;
      const int L = std::max(lens[pc.b], 0);
      if (!(0 <= pc.st && pc.st < pc.en && pc.en <= L)) return "piece outside its sequence";
      if (pc.st % kSchedTile) return "piece start off the tile grid";
      if (pc.slot < 0 || pc.slot >= S) return "slot out of range";
      if (pc.slot != next_slot[pc.b]) return "slots not consecutive in token order";
      ++next_slot[pc.b];
      for (int t = pc.st; t < pc.en; ++t) {
        if (covered[pc.b][t]) return "token covered twice";
        covered[pc.b][t] = 1;
      }
      if (pc.en == L) {   // the last piece marks the slots after its own (none when it holds slot S - 1)
        if (pc.fill_from != pc.slot + 1) return "last piece does not mark the unused slots";
        ++lasts[pc.b];
      } else if (pc.fill_from != S) {
        return "unused slots marked by a piece that is not the last";
      }
      mine += (pc.en - pc.st + kSchedTile - 1) / kSchedTile;
    }
    *max_tiles = std::max(*max_tiles, mine);
    if (mine > quota) return "pair above its quota";
  }
  for (int b = 0; b < B; ++b) {
    for (size_t t = 0; t < covered[b].size(); ++t)
      if (!covered[b][t]) return "token not covered";
    if (lens[b] > 0 && lasts[b] != 1) return "no last piece";
  }
  return "";
}

int main() {
  int B, S, pairs;
  while (std::scanf("%d %d %d", &B, &S, &pairs) == 3) {
    std::vector<int32_t> lens(B);
    for (int b = 0; b < B; ++b)
      if (std::scanf("%d", &lens[b]) != 1) return 2;
    long long mt = 0, ideal = 0, np = 0;
    int split = 0;
    const std::string err = run_case(B, S, pairs, lens, &mt, &ideal, &np, &split);
    if (err.empty())
      std::printf("ok %lld %lld %lld %d\n", mt, ideal, np, split);
    else
      std::printf("fail %s\n", err.c_str());
  }
  return 0;
}
