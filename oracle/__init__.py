"""Float64 CPU oracle for the exact attention forward.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check in
``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import this package.  The CUDA library never calls it and it
never calls the CUDA library: the two share no code.  The only thing both sides
consume is the seeded input generator, which lives in its own module and holds
none of the attention arithmetic.

Pages this oracle follows (cited by title and section):

* "Inside FlashAttention-3：面向 Hopper 架构的 IO-Aware 精确注意力机制深度解析"
  (the FA-3 page), section 二 "核心算法：Two-Level 在线 Softmax 的再回顾" — the
  running-max / running-sum / rescaled-accumulator recurrence; section 十
  "总结" — the method does not change the mathematical definition of attention.
* The FA-3 page, section 7.2 "cuDNN 集成" — variable-length sequences as
  ragged tensors (``attention_varlen_f64``: one attention problem per packed
  sequence).
* The FA-3 page, section 7.3 "BF16 / FP8 支持" — e4m3 inputs with fp32
  statistics (``oracle.fp8``: the attention of the encoded values, an e4m3
  decoder written from the format's bit fields, and the size of the error that
  rounding P to e4m3 adds).
* The FA-2 page, sections "warp之间怎样减少通信" and "训练与部署 切分与归约的反向
  一致性" — the training backward, dQ, dK, dV with dK and dV accumulated across
  query rows, and a printed score gradient (``oracle.backward``).
* "AI 大模型之 FlashAttention_02" (the FA-2 page), section 3.1 and 4.1 — exact
  softmax attention, O(S²d); section "工程实操 沿键切分的归约与沿查询切分的区别" —
  split partial states (m, l, u) and the merge that rescales by exp(m_b − M).

Every function is pinned by ``tests/test_oracle.py`` against values printed on
the pages, closed forms, invariants, a library routine, brute force and (for
the e4m3 error scale) a simulation of the error model it states.
"""

from .attention import (  # noqa: F401
    attention_f64,
    attention_varlen_f64,
    attention_rows_f64,
    scores_f64,
    online_softmax_state_f64,
    split_states_f64,
    merge_states_f64,
    normalise_then_average_f64,
)
from . import backward, fp8  # noqa: F401,E402
