"""CPU fp64 oracle for exact attention (forward and backward) and the pages' IO model.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link anything in this package: only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code, tables or helpers with the CUDA library, and the CUDA library
never produces an input or an expected value for it.

Sources, cited by page title and section throughout:

* [T]  blog.teqners.com, "13% more FLOPs, 5.7x faster: how FlashAttention's
       online softmax keeps the N x N matrix out of HBM"
* [V]  blog.vikramsamal.com, "FlashAttention and the art of GPU mechanics"
* [L]  lensaml.com, "FlashAttention" explainer (Steps 1-6 and the FAQ)

Pins (tests/test_oracle_*.py) tie every function here to something other than
itself: the worked example and printed numbers of [L], closed forms, invariants,
PyTorch's own fp64 ``scaled_dot_product_attention`` and autograd, SciPy's
``logsumexp``/``softmax``, and central finite differences.
"""

from .attention import (  # noqa: F401
    attention_backward,
    attention_backward_head,
    attention_backward_head_rows,
    attention_forward,
    attention_forward_head_rows,
    attention_forward_tiled,
    online_softmax_trace,
    scores,
    softmax_three_pass,
)
from .decode import attention_forward_rect, merge_partials, split_bounds, split_partials  # noqa: F401
from . import dropout  # noqa: F401
from . import fp8  # noqa: F401
from . import io_model  # noqa: F401
