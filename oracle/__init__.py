"""Float64 CPU oracle of the SSSL / GQA / QK-norm attention block.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the library. It shares no
code with the CUDA path.
"""
from .attention import *  # noqa: F401,F403
from .attention import __all__ as _attention_all
from .block import *  # noqa: F401,F403
from .block import __all__ as _block_all

__all__ = list(_attention_all) + list(_block_all)
