"""Oracle for sharded ring attention: plain, slow, float64, CPU only.

THIS PACKAGE IS TEST INFRASTRUCTURE.  Only the tests, the smoke check and the
benchmark's CPU-baseline / reference arm may import it.  The CUDA library
never calls it and it never calls the CUDA library; the two share no code.

What it computes, and where each part comes from:
  * ``layout``      -- sharding shapes -> shard offsets; the zigzag
                       re-partition -> natural position of every buffer row.
                       (ShardTensor summary, section 2 "sharding shapes";
                       TSP summary, section 2, attention layer, zigzag.)
  * ``attention``   -- full softmax attention by its definition, the
                       ring-attention formulation (each query shard meets
                       every KV shard, partials merged by the log-sum-exp
                       rule), and the textbook backward.  (ShardTensor
                       summary, section 4, ring attention benchmark; TSP
                       summary, section 2, all-gathered K/V + FlashAttention,
                       which computes the same function as full attention.)
  * ``bruteforce``  -- pure-Python loops for tiny inputs.
  * ``projection``  -- the linear layers on either side of the attention, by
                       their definition and by the broadcast schedule of the
                       pages (TSP summary, section 2, attention layer: every
                       rank projects its sequence shard with each packed
                       W_Q, W_K, W_V, W_O shard in turn).
  * ``mlp``         -- the gated MLP by its definition and by the pages'
                       ring schedule (TSP summary, section 2, gated MLP
                       layer: W1, W2, W3 shards travel round the ring while
                       every rank adds up its partial outputs).
  * ``halo``        -- 2-D convolution of a row-sharded image with uneven
                       shards: the halo exchange (neighbouring rows taken
                       from the shards that own them) and the local
                       convolutions, equal to the layer on the whole image
                       (ShardTensor summary, section 2, communication: halo
                       exchange for convolution and normalisation).
  * ``norm``        -- group normalisation of a row-sharded image: local
                       statistics, their all-reduce, local normalisation
                       (the same passage: collectives for normalisation).

All floating point is float64 on the values the caller passes (for bf16 inputs
the caller passes the bf16-rounded values).  Every function is pinned by tests
that do not re-type its formula: a library attention routine, closed forms,
invariants the pages fix (sharded == unsharded, zigzag-causal == causal) and
finite differences.
"""
from . import layout, attention, bruteforce, projection, mlp, halo, norm  # noqa: F401
