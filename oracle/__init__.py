"""CPU oracle for the shape-batched Newton-Schulz hot path.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call, link
or execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code with the CUDA library (``newton_schulz_shape_gb300``) and imports
nothing from it.

Modules
-------
``ns``        quintic Newton-Schulz in float64 (numpy), plus a pure-Python
              loop version for tiny inputs.
``planning``  2-D views, the Newton-Schulz cost estimate, candidate holders,
              greedy LPT owner assignment and ``params_by_home``.
``routing``   row-shard pack/unpack (shard -> home and back) and the
              flat-buffer OwnerGatherPlan / OwnerScatterPlan metadata seen
              from one rank.

Sources: the Megatron-Core API pages ``core.optimizer.layer_sharded_a2a`` and
``core.distributed.fsdp.src.megatron_fsdp.experimental.owner_planning``, and
the Megatron-LM GitHub issue "[GTP][Muon] Optimize Muon step performance"
(#6720). Each function names the entry it follows.

Pinning status: every function here is pinned by a ``-m "not gpu"`` test
against the pages' worked example, closed forms, library routines or brute
force. The trace-ridge term of ``ns.newton_schulz`` (``ridge > 0``) is pinned
to the singular-value closed form of its reading (A <- A + ridge * tr(A)/m * I
before B is formed); the placement and scale themselves are that reading, as
the issue names a trace ridge without giving its form.
"""

from . import ns, planning, routing  # noqa: F401
