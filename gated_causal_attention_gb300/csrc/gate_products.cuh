// gate_products.cuh -- how the path product is assembled from the gate-prep outputs.
//
// "Resolvent Operator", section "Object", path-product row: G_ij = prod_{k=j+1..i} a_k.
// For a query row i in block QB and a key j in an earlier block KB the product splits at
// the block edges:
//     G_ij = prefix_i * C(QB,KB) * suffix_j,   C(QB,KB) = prod_{KB < b < QB} carry_b,
// where C starts at 1 for KB = QB-1 and takes one more block total per step as KB
// descends. Inside one block the product is taken explicitly, one gate at a time, from
// j = i down. Every step is a multiplication -- no logarithm, no division by a prefix --
// so a closed gate (a_k = 0) gives an exact zero wherever it lies on the path.
// The head kernel and the debug export both use these helpers, so the export shows
// exactly the products the head kernel forms.
#pragma once

#include "common.cuh"

namespace rs {

// C(QB, KB-1) from C(QB, KB): fold in the total of block KB.
__device__ __forceinline__ cplx carry_step(cplx C, cplx block_total) { return cmul(C, block_total); }

// Scale of key j under carry C: C * suffix_j (the factor applied to V_j).
__device__ __forceinline__ cplx key_scale(cplx C, cplx suffix_j) { return cmul(C, suffix_j); }

// Off-diagonal path product: prefix_i * (C * suffix_j).
__device__ __forceinline__ cplx offdiag_product(cplx prefix_i, cplx key_scale_j)
{
    return cmul(prefix_i, key_scale_j);
}

// Inside a block: G_{i,j} = G_{i,j+1} * a_{j+1}, starting from G_{i,i} = 1.
__device__ __forceinline__ cplx diag_step(cplx G, cplx a_next) { return cmul(G, a_next); }

}  // namespace rs
