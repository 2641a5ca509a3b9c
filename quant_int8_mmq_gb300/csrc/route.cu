// route.cu -- host-side kernel choice for M above the few-token range and the registry
// of packed q6_K weights' fold state.  See route.h.
#include "route.h"

#include <cstdint>
#include <mutex>
#include <unordered_map>

namespace mmq {
namespace {

struct PackedKey {
    int dev;
    uintptr_t addr;
    bool operator==(const PackedKey& o) const { return dev == o.dev && addr == o.addr; }
};
struct PackedKeyHash {
    size_t operator()(const PackedKey& k) const
    {
        return std::hash<uintptr_t>()(k.addr) ^ (static_cast<size_t>(k.dev) * 0x9E3779B97F4A7C15ull);
    }
};
struct PackedInfo {
    int type, od, id, fold;
};

std::mutex g_mu;
std::unordered_map<PackedKey, PackedInfo, PackedKeyHash>& registry()
{
    static std::unordered_map<PackedKey, PackedInfo, PackedKeyHash> m;
    return m;
}

// Launch-time estimate of a tile kernel in microseconds on GB300 (only the comparison
// of the two kernels matters).  A persistent launch of T tiles on nsm SMs runs F rounds
// of whole tiles and, where the kernels' split rule applies (every tile when 2T <= nsm,
// else a last round of at most nsm/2 tiles, and only with at least two super-blocks),
// one round of K-halves (S = 1):  t = a + F (f + b nsb) + S (g + h nsb),  nsb = id/256.
// The constants are a least-squares fit, on relative error, to CUDA-graph timings of
// both kernels on GB300 (q4_K and scale-folded q6_K; 148 cases, M = 129..2048,
// od = 2048..32000, id = 512..14336, 4 rotated weight copies).  Over those cases the
// pick was never more than 3.4 % slower than the faster kernel; "super-block kernel
// when its tiles fill every SM once" had been up to 40 % slower.
struct RoundCost {
    double a, f, b, g, h;
};
constexpr RoundCost CHUNK_COST{3.35, 2.91, 1.80, 6.16, 0.93};   // 128 x 128 tiles
constexpr RoundCost SB_COST{3.45, 4.42, 2.79, 11.95, 1.40};     // 128 x 256 tiles

double estimate_us(const RoundCost& c, long long tiles, int nsb, int nsm)
{
    long long full = 0;
    int split_round = 0;
    if (nsb >= 2 && 2 * tiles <= nsm) {
        split_round = 1;
    } else {
        full = tiles / nsm;
        const long long rem = tiles % nsm;
        if (rem > 0) {
            if (nsb >= 2 && full > 0 && 2 * rem <= nsm)
                split_round = 1;
            else
                ++full;
        }
    }
    return c.a + static_cast<double>(full) * (c.f + c.b * nsb) + split_round * (c.g + c.h * nsb);
}

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace

void note_packed(int dev, const void* packed, int type, int od, int id, int fold)
{
    const PackedKey k{dev, reinterpret_cast<uintptr_t>(packed)};
    std::lock_guard<std::mutex> lock(g_mu);
    if (fold < 0)
        registry().erase(k);
    else
        registry()[k] = PackedInfo{type, od, id, fold};
}

int packed_fold_state(int dev, const void* packed, int type, int od, int id)
{
    const PackedKey k{dev, reinterpret_cast<uintptr_t>(packed)};
    std::lock_guard<std::mutex> lock(g_mu);
    const auto it = registry().find(k);
    if (it == registry().end())
        return -1;
    const PackedInfo& p = it->second;
    return (p.type == type && p.od == od && p.id == id) ? p.fold : -1;
}

bool prefer_superblock(int type, int od, int id, int M, int nsm, int fold)
{
    // q6_K in two tiles: the chunk kernel at every M.  Its promotion (one FMA per
    // accumulator element per chunk) leaves the tensor pipe room for the second tile's
    // MMAs, while the super-block kernel's tensor work doubles: on GB300 the chunk
    // kernel was 14 to 58 % faster over M = 129..3314 on four shapes.
    if (type == 14 && fold == 0)
        return false;
    if (nsm <= 0)
        nsm = 1;
    const long long mt = cdiv(M, 128);
    const int nsb = id / 256;
    return estimate_us(SB_COST, mt * cdiv(od, 256), nsb, nsm) < estimate_us(CHUNK_COST, mt * cdiv(od, 128), nsb, nsm);
}

}  // namespace mmq
