// Decode attention over the paged KV cache: what the partition kernels and
// the split-K reduce compute, and the workspace they share.
//
// What is computed ("19.2 KV Cache 系统化管理" §19.2.3 paged_attention;
// "KV Cache：长上下文为什么吃显存" §01/§02): for sequence s and query head h
// (KV head j = h / G), out = softmax(scale * q . K_j[0:L]) V_j[0:L], with K/V
// rows found through the block table (token t -> block bt[s][t / K], offset
// t % K).  Scores and weights are kept in the base-2 domain
// (x = scale * log2(e) * q.k, weight = 2^(x - max)), which is the same
// softmax.  Every kernel keeps the running maximum m, the running sum l and
// the unnormalised output o of the page's block loop; partial states of one
// (s, h) are merged by attn_reduce_kernel with
//   M = max m_p,  l = sum l_p 2^(m_p - M),  out = sum o_p 2^(m_p - M) / l.
//
// Workspace (per launch batch): partial states live in slots, slot x holding
// (m, l) at ml[x * H_q + h] and o at o[(x * H_q + h) * D]; meta[r] =
// (base1, n1, base2, n2) says that output row r (a sequence, or a query row)
// has its partials in slots base1 .. base1 + n1 - 1 and base2 .. base2 + n2 - 1
// (n1 + n2 <= 1: the partition kernel wrote the output itself).
//   CUDA-core kernel, multi-query launches: row r's partial p in slot
//     r * pmax + p;
//   tensor-core decode kernel: the partition of CTA i over unit u in slot
//     i + u (a unit's CTAs are consecutive, so are its slots); a shared unit
//     keeps one region of slots per member sequence.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

struct Workspace {
  int4* meta;
  float2* ml;
  float* o;
  int pmax;
};

}  // namespace pkv
