// Host interface of the Goldfish-loss kernels (goldfish.cu): the hashed
// token mask, the masked cross-entropy with its gradient over bf16 logits,
// and the fixed-order mean.  The C entry point that validates arguments and
// calls these is axonn_goldfish_ce in axonn_fc.cu.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace axonn {

struct GoldfishArgs {
  const uint16_t* logits;  // bf16 [T x V], row stride ld_logits elements
  int64_t ld_logits;
  const int32_t* input_ids;  // [batch x seq]
  const int32_t* labels;     // [batch x seq]
  int64_t batch, seq, vocab;
  int32_t k, h;
  uint8_t* keep;       // [T]
  float* token_loss;   // [T]
  float* loss;         // [1]
  int32_t* kept;       // [1]
  uint16_t* dlogits;   // bf16 [T x V] or null, row stride ld_dlogits
  int64_t ld_dlogits;
  uint64_t timeout_ns;
  int32_t inject;  // 1: the rows kernel withholds every copy (a test of the bounded waits)
};

// Largest vocabulary the entry point accepts (8 x 49152 tokens).
constexpr int64_t kGoldfishMaxVocab = 8 * 49152;

// Whether a vocabulary of `vocab` tokens is in [1, kGoldfishMaxVocab].
bool goldfish_vocab_supported(int64_t vocab);

// The three launches (mask and count, rows, mean) on `stream`; the rows
// kernel runs one persistent CTA on each of the `sms` SMs (fewer for fewer
// rows).
cudaError_t goldfish_launch(const GoldfishArgs& a, int sms, cudaStream_t stream);

// Reads (and clears if set) the device error word of these kernels.
cudaError_t goldfish_take_status(unsigned long long* word, cudaStream_t stream);

}  // namespace axonn
