// packer.cu -- host-side sequence packing (declared in include/varlen_ssm.h).
//
// The article "Shanghai AI Lab: packed variable-length Mamba training",
// section 结论与讨论, names two ways to fill packs of a fixed token budget:
// its own, which takes sequences in arrival order and seals a pack when the
// next sequence does not fit (19.1 % padding on its pretraining data), and a
// local greedy one, which sorts a portion of the pending sequences first and
// then packs greedily (down to 0.46 %), at the price of the sort.  Both run
// here on the calling thread, on host arrays; the packs they return are what
// a data loader turns into one cu_seqlens per pack.
#include <algorithm>
#include <cstdio>
#include <numeric>
#include <vector>

#include "kernels.h"
#include "varlen_ssm.h"

using namespace vssm;

namespace {

int fail_arg(const char* fmt, long long a = 0, long long b = 0) {
  char buf[256];
  snprintf(buf, sizeof(buf), fmt, a, b);
  return record_error(VSSM_ERR_ARG, buf);
}

}  // namespace

extern "C" int varlen_pack_sequences(const int32_t* lengths, int32_t num_seqs, int32_t pack_size,
                                     int32_t method, int32_t window, int32_t* order,
                                     int32_t* pack_offsets, int32_t* num_packs, double* padding_rate) {
  if (num_seqs < 0) return fail_arg("num_seqs %lld is negative", num_seqs);
  if (pack_size <= 0) return fail_arg("pack_size %lld is not positive", pack_size);
  if (method != VSSM_PACK_SEQUENTIAL && method != VSSM_PACK_LOCAL_GREEDY)
    return fail_arg("unknown packing method %lld", method);
  if (method == VSSM_PACK_LOCAL_GREEDY && window <= 0) return fail_arg("window %lld is not positive", window);
  if (!num_packs || !padding_rate || !pack_offsets || (num_seqs > 0 && (!lengths || !order)))
    return record_error(VSSM_ERR_ARG, "NULL lengths, order, pack_offsets, num_packs or padding_rate");
  int64_t used_total = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    if (lengths[i] < 0) return fail_arg("length %lld of sequence %lld is negative", lengths[i], i);
    if (lengths[i] > pack_size)
      return fail_arg("sequence %lld is longer than a pack (%lld tokens)", i, lengths[i]);
    used_total += lengths[i];
  }

  int32_t np = 0, k = 0;  // packs sealed, entries of `order` written
  pack_offsets[0] = 0;
  if (method == VSSM_PACK_SEQUENTIAL) {
    int64_t used = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
      if (k > pack_offsets[np] && used + lengths[i] > pack_size) {  // seal: the next one does not fit
        pack_offsets[++np] = k;
        used = 0;
      }
      order[k++] = i;
      used += lengths[i];
    }
    if (k > pack_offsets[np]) pack_offsets[++np] = k;
  } else {
    std::vector<int32_t> idx;
    std::vector<std::vector<int32_t>> packs;
    std::vector<int64_t> room;
    for (int32_t w0 = 0; w0 < num_seqs; w0 += window) {
      const int32_t w1 = std::min<int64_t>((int64_t)w0 + window, num_seqs);
      idx.resize(w1 - w0);
      std::iota(idx.begin(), idx.end(), w0);
      // longest first; equal lengths keep their arrival order
      std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return lengths[a] > lengths[b]; });
      packs.clear();
      room.clear();
      for (const int32_t i : idx) {  // first fit among this window's packs
        size_t p = 0;
        while (p < packs.size() && room[p] < lengths[i]) ++p;
        if (p == packs.size()) {
          packs.emplace_back();
          room.push_back(pack_size);
        }
        packs[p].push_back(i);
        room[p] -= lengths[i];
      }
      for (const auto& p : packs) {  // sealed in the order they were opened
        for (const int32_t i : p) order[k++] = i;
        pack_offsets[++np] = k;
      }
    }
  }
  *num_packs = np;
  *padding_rate = np > 0 ? 1.0 - (double)used_total / ((double)np * (double)pack_size) : 0.0;
  return VSSM_OK;
}
