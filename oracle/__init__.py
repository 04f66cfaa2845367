"""CPU oracle for wave-index tripartite decode attention and its segmented
spherical k-means index build.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  The product path (the CUDA
library and its Python binding) never imports, calls or falls back to it, and
it shares no code with that path: it depends on NumPy alone.

Parity status per function is stated in ``wave_index``'s module docstring.
"""

from .wave_index import *  # noqa: F401,F403
