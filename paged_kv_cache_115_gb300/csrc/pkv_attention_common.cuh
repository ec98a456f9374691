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
// Workspace layout (per launch batch of sequences, Pmax partials per seq):
//   int    nparts[S]                   partials written for s (0: empty seq,
//                                      1: output already final)
//   float2 ml[S][Pmax][H_q]            (m, l) of each partial
//   float  o [S][Pmax][H_q][D]         unnormalised partial outputs
#pragma once

#include "pkv_device.cuh"

namespace pkv {

struct Workspace {
  int* nparts;
  float2* ml;
  float* o;
  int pmax;
};

}  // namespace pkv
