"""Plain CPU oracle of the autoregressive-denoising DiT wave path.

TEST INFRASTRUCTURE, not product code.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
It shares no code with the CUDA library (``autoregressive_denoising_dit_gb300``)
and neither imports the other; the seeded inputs both consume come from the
arithmetic-free ``synth`` module.

Modules: ``model`` (block math), ``schedule`` (task DAG, wave plan, KV ring,
brute force), ``runner`` (streams, chunks, steps, wave and sequential order).

Parity status: every function is pinned by a test in ``tests/test_oracle_*``
(brute-force loops, closed forms, invariants, the pages' worked pipeline
example); see the pin list in each test module.
"""
from . import model, schedule, runner  # noqa: F401
from .runner import OracleRunner  # noqa: F401
