// Arguments of the appends of a decode step, shared by the kernels that run them.  Internal to
// the library.
#pragma once

#include <stdint.h>

#include "tq_internal.h"

namespace tq {

// The appends of a decode step: the new key (product code) and value (MSE code) of every
// (batch, KV head), at position pos[b] of the caches.
struct AppendKV {
  const void* k_new;           // [B][Hkv][128] of dtype
  const void* v_new;
  int dtype;
  const int* pos;              // device int32[B]
  int* lens_out;               // device int32[B] or null: receives pos[b] + 1
  int Hkv, cap;
  uint8_t* kidx;               // key cache (product code)
  uint8_t* ksgn;
  float* kxn;
  float* krn;
  uint8_t* vidx;               // value cache (MSE code)
  float* vxn;
  const float* kpiT;           // Πᵀ and Mᵀ of the key codec, Πᵀ of the value codec
  const float* kmT;
  const float* vpiT;
  tq_levels klv, vlv;
  int kbits, vbits;            // index bits
  int v_nibbles;               // value codes nibble-packed (4 bits)
  int shared_pi;               // the two codecs hold the same Π: kpiT serves the values too
  tq_rowmap kmap, vmap;        // the caches' row maps (flat, or block tables)
};

}  // namespace tq
