"""CPU oracle for mean-pooled, block-routed, block-sparse attention.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
float64 restatement of the definitions given on four pages:

* "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" (maple.link) -- 3D tiling,
  mean pooling, the routing matrix E, per-row TopK, block-sparse attention,
  and the gated coarse branch softmax(E) V_bar.
* "NSA 算子解析（Torch/Tilelang）" (devpress.csdn.net) -- the selected-attention
  branch with caller-supplied block indices/counts and GQA.
* "MSA 为什么采用 KV-outer Sparse Attention Forward" (notes.kuangjux.top) -- the
  reverse index, the K1 partial pass and the K2 log-sum-exp combine.
* "深度解读|Spark-H3：从注意力几何到稀疏内核代码" (jefxiong.cn) -- the
  exact-plus-summary mixture with the +log(m) mass term, the Reweight
  summaries (weighted key and value with a log-mass bias at a representative
  query) and the Reblock layout (second-moment metric, equal-capacity
  hierarchical partition).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never imports it, links it or calls it, and the two share no code: the
oracle takes plain numpy arrays, the library takes device pointers.

Every function works on one (batch, head) slice unless it says otherwise and
computes in float64 with numpy; a matmul, a sort and ``exp``/``log`` are the
only library primitives used.

Parity pins: every public function here is pinned by ``tests/test_oracle_pins.py``
to values printed on the pages, closed forms, library routines (``torch``'s
float64 ``scaled_dot_product_attention`` on CPU) or brute force on tiny inputs.
"""

from .tiling import (  # noqa: F401
    num_blocks, token_index, tile_3d, tile_prefix, tile_permuted, index_map, budget, tile_segments,
)
from .pool import pool_blocks  # noqa: F401
from .route import routing_scores, topk_row, route, route_grouped, near_tie_rows  # noqa: F401
from .attention import (  # noqa: F401
    softmax_attention, dense_attention, block_sparse_attention, summary_attention,
    nsa_selected_attention, pair_counts,
)
from .kvouter import (  # noqa: F401
    reverse_index, schedule_chunks, kvouter_partials, combine_partials,
)
from .spark import bf16_round, reweight_anchor, reweight_summary, reweight_summaries  # noqa: F401
from .coarse import coarse_attention, coarse_output  # noqa: F401
from .reblock import (  # noqa: F401
    second_moment, metric_factor, unit_features, split_node, partition, reblock_layout, attention_mass_recall,
)
