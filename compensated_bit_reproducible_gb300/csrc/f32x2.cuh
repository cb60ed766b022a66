// Two float lanes in one 64-bit register (x in the low word, y in the high
// word) and the packed operations on them.
//
// add.rn.f32x2 and sub.rn.f32x2 are two independent IEEE round-to-nearest
// operations in one instruction, subnormals kept: the bits of two scalar
// operations, for half the issue slots.  Products are not packed here: a
// packed multiply feeding a packed add was measured to be contracted into a
// fused multiply-add on GB300 (about 20% of random operand pairs differed
// from the two roundings), even with FMA contraction disabled, while scalar
// products packed into a packed add kept both roundings in every pair.
#pragma once
#include <cstdint>

namespace repro {

typedef unsigned long long F2;

__device__ __forceinline__ F2 pk2(float x, float y) {
  F2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void up2(F2 v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ F2 add2(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ F2 sub2(F2 a, F2 b) {
  F2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

}  // namespace repro
