// Optional per-kernel timing of the library's own launches (off by default):
// when enabled, each launch is bracketed by CUDA events on its stream and
// the elapsed times are accumulated per kernel name until read.
#pragma once

#include <cuda_runtime.h>

namespace moe {
namespace prof {

bool enabled();
// Returns a token to pass to end(); no-op (returns -1) when disabled.
int begin(const char* name, cudaStream_t s);
void end(int token, cudaStream_t s);

struct Scope {
  int tok;
  cudaStream_t s;
  Scope(const char* name, cudaStream_t st) : tok(begin(name, st)), s(st) {}
  ~Scope() { end(tok, s); }
};

}  // namespace prof
}  // namespace moe
