// prefix_cache.cpp -- host-side prefix cache: the hash chain of the tutorial
// page "LLM 推理服务引擎深度拆解", section 4 (prefix caching), sections 4.2
// and 4.3.
//
// A prompt is cut into full blocks of block_size tokens.  Block i's key is
//   sha256( parent + tokens + extra )[first 32 hex digits]
// where parent is block i-1's key ("ROOT" for block 0), tokens is the block's
// token ids written in decimal and joined by commas, and extra is a caller
// string (for example to tell apart images behind equal placeholder ids).
// The parent term makes a key name a whole prefix, so the longest cached
// prefix ends at the first key the table does not hold.  A lookup returns the
// keys of every full block of the prompt (hits counted up to the first miss
// only) so that one insert can cache the whole prompt.  The table maps
// key -> physical block id, holds at most capacity entries and evicts the
// least recently used key; a lookup touches the keys it hits and counts one
// hit (some prefix found) or one miss; insert adds the keys it does not hold
// and touches every key of the chain.
//
// SHA-256 is written here from its definition (FIPS 180-4): 64 rounds over
// 512-bit blocks, big-endian words, message padded with 0x80, zeros and the
// 64-bit bit length.  Round constants: first 32 bits of the fractional parts
// of the cube roots of the first 64 primes; initial state: the same of the
// square roots of the first 8 primes.
#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "pd_attn.h"

namespace {

constexpr uint32_t kRound[64] = {
    0x428a2f98u, 0x71374491u, 0xb5c0fbcfu, 0xe9b5dba5u, 0x3956c25bu, 0x59f111f1u, 0x923f82a4u,
    0xab1c5ed5u, 0xd807aa98u, 0x12835b01u, 0x243185beu, 0x550c7dc3u, 0x72be5d74u, 0x80deb1feu,
    0x9bdc06a7u, 0xc19bf174u, 0xe49b69c1u, 0xefbe4786u, 0x0fc19dc6u, 0x240ca1ccu, 0x2de92c6fu,
    0x4a7484aau, 0x5cb0a9dcu, 0x76f988dau, 0x983e5152u, 0xa831c66du, 0xb00327c8u, 0xbf597fc7u,
    0xc6e00bf3u, 0xd5a79147u, 0x06ca6351u, 0x14292967u, 0x27b70a85u, 0x2e1b2138u, 0x4d2c6dfcu,
    0x53380d13u, 0x650a7354u, 0x766a0abbu, 0x81c2c92eu, 0x92722c85u, 0xa2bfe8a1u, 0xa81a664bu,
    0xc24b8b70u, 0xc76c51a3u, 0xd192e819u, 0xd6990624u, 0xf40e3585u, 0x106aa070u, 0x19a4c116u,
    0x1e376c08u, 0x2748774cu, 0x34b0bcb5u, 0x391c0cb3u, 0x4ed8aa4au, 0x5b9cca4fu, 0x682e6ff3u,
    0x748f82eeu, 0x78a5636fu, 0x84c87814u, 0x8cc70208u, 0x90befffau, 0xa4506cebu, 0xbef9a3f7u,
    0xc67178f2u};
constexpr uint32_t kInit[8] = {0x6a09e667u, 0xbb67ae85u, 0x3c6ef372u, 0xa54ff53au,
                               0x510e527fu, 0x9b05688cu, 0x1f83d9abu, 0x5be0cd19u};

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void sha256_block(uint32_t st[8], const unsigned char* p) {
    uint32_t w[64];
    for (int i = 0; i < 16; ++i)
        w[i] = (uint32_t(p[4 * i]) << 24) | (uint32_t(p[4 * i + 1]) << 16) |
               (uint32_t(p[4 * i + 2]) << 8) | uint32_t(p[4 * i + 3]);
    for (int i = 16; i < 64; ++i) {
        const uint32_t s0 = rotr(w[i - 15], 7) ^ rotr(w[i - 15], 18) ^ (w[i - 15] >> 3);
        const uint32_t s1 = rotr(w[i - 2], 17) ^ rotr(w[i - 2], 19) ^ (w[i - 2] >> 10);
        w[i] = w[i - 16] + s0 + w[i - 7] + s1;
    }
    uint32_t a = st[0], b = st[1], c = st[2], d = st[3], e = st[4], f = st[5], g = st[6],
             h = st[7];
    for (int i = 0; i < 64; ++i) {
        const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
        const uint32_t ch = (e & f) ^ (~e & g);
        const uint32_t t1 = h + S1 + ch + kRound[i] + w[i];
        const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
        const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
        const uint32_t t2 = S0 + maj;
        h = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + t2;
    }
    st[0] += a; st[1] += b; st[2] += c; st[3] += d;
    st[4] += e; st[5] += f; st[6] += g; st[7] += h;
}

// Lower-case hex digest of msg.
std::string sha256_hex(const std::string& msg) {
    uint32_t st[8];
    std::memcpy(st, kInit, sizeof(st));
    const size_t n = msg.size();
    const unsigned char* m = reinterpret_cast<const unsigned char*>(msg.data());
    size_t off = 0;
    for (; off + 64 <= n; off += 64) sha256_block(st, m + off);
    unsigned char tail[128] = {};
    const size_t rest = n - off;
    std::memcpy(tail, m + off, rest);
    tail[rest] = 0x80;
    const size_t tail_len = rest + 1 + 8 <= 64 ? 64 : 128;
    const uint64_t bits = uint64_t(n) * 8;
    for (int i = 0; i < 8; ++i) tail[tail_len - 1 - i] = (unsigned char)(bits >> (8 * i));
    for (size_t o = 0; o < tail_len; o += 64) sha256_block(st, tail + o);
    static const char* hex = "0123456789abcdef";
    std::string out(64, '0');
    for (int i = 0; i < 8; ++i)
        for (int k = 0; k < 8; ++k) out[size_t(8 * i + k)] = hex[(st[i] >> (28 - 4 * k)) & 0xf];
    return out;
}

constexpr int kKeyChars = 32;

std::string block_key(const std::string* parent, const int32_t* tokens, int n,
                      const char* extra) {
    std::string msg = parent ? *parent : std::string("ROOT");
    for (int i = 0; i < n; ++i) {
        if (i) msg.push_back(',');
        msg += std::to_string(tokens[i]);
    }
    if (extra) msg += extra;
    return sha256_hex(msg).substr(0, kKeyChars);
}

}  // namespace

struct pd_pc {
    int capacity;
    int block_size;
    std::unordered_map<std::string, int32_t> table;
    std::list<std::string> lru;    // front = least recently used
    std::unordered_map<std::string, std::list<std::string>::iterator> where;
    int64_t hits = 0, misses = 0;

    void touch(const std::string& k) {
        auto it = where.find(k);
        if (it != where.end()) lru.erase(it->second);
        lru.push_back(k);
        where[k] = std::prev(lru.end());
    }
};

extern "C" {

pd_pc* pd_pc_create(int capacity_blocks, int block_size) {
    if (capacity_blocks < 1 || block_size < 1) return nullptr;
    pd_pc* pc = new (std::nothrow) pd_pc();
    if (!pc) return nullptr;
    pc->capacity = capacity_blocks;
    pc->block_size = block_size;
    return pc;
}

void pd_pc_destroy(pd_pc* pc) { delete pc; }

pd_status pd_pc_lookup(pd_pc* pc, const int32_t* token_ids, int n, const char* extra,
                       int* hit_tokens, char* chain_out, int32_t* hit_blocks_out,
                       int* n_chain) {
    if (!pc || n < 0 || (n > 0 && !token_ids) || !hit_tokens || !n_chain)
        return PD_ERR_INVALID_ARG;
    const int S = pc->block_size;
    const int nfull = n / S;
    if (nfull > 0 && !chain_out) return PD_ERR_INVALID_ARG;
    try {
        std::string parent;
        int hit = 0, nc = 0;
        bool in_prefix = true;
        for (int i = 0; i + S <= n; i += S) {
            const std::string k = block_key(nc ? &parent : nullptr, token_ids + i, S, extra);
            std::memcpy(chain_out + size_t(nc) * (kKeyChars + 1), k.c_str(), kKeyChars + 1);
            ++nc;
            if (in_prefix) {
                auto it = pc->table.find(k);
                if (it == pc->table.end()) {
                    in_prefix = false;               // no later block can hit
                } else {
                    if (hit_blocks_out) hit_blocks_out[hit / S] = it->second;
                    hit += S;
                    pc->touch(k);
                }
            }
            parent = k;
        }
        if (hit) pc->hits += 1;
        else pc->misses += 1;
        *hit_tokens = hit;
        *n_chain = nc;
    } catch (...) {
        return PD_ERR_INVALID_ARG;
    }
    return PD_OK;
}

pd_status pd_pc_insert(pd_pc* pc, const char* chain, int n_chain, const int32_t* block_ids,
                       int32_t* evicted_out, int* n_evicted) {
    if (!pc || n_chain < 0 || (n_chain > 0 && (!chain || !block_ids))) return PD_ERR_INVALID_ARG;
    int ne = 0;
    try {
        for (int i = 0; i < n_chain; ++i) {
            const char* c = chain + size_t(i) * (kKeyChars + 1);
            const std::string k(c, strnlen(c, kKeyChars));
            if (!pc->table.count(k)) {
                if (int(pc->table.size()) >= pc->capacity) {
                    const std::string victim = pc->lru.front();
                    pc->lru.pop_front();
                    pc->where.erase(victim);
                    auto v = pc->table.find(victim);
                    if (v != pc->table.end()) {
                        if (evicted_out) evicted_out[ne] = v->second;
                        ++ne;
                        pc->table.erase(v);
                    }
                }
                pc->table[k] = block_ids[i];
            }
            pc->touch(k);
        }
    } catch (...) {
        return PD_ERR_INVALID_ARG;
    }
    if (n_evicted) *n_evicted = ne;
    return PD_OK;
}

int pd_pc_size(const pd_pc* pc) { return pc ? int(pc->table.size()) : -1; }
int64_t pd_pc_hits(const pd_pc* pc) { return pc ? pc->hits : -1; }
int64_t pd_pc_misses(const pd_pc* pc) { return pc ? pc->misses : -1; }

}  // extern "C"
