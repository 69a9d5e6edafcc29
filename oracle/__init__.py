"""Oracle for the virtual-rank collectives -- TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded CPU model of N ranks exchanging messages step by
step, written twice from the three source pages: as a C++17 program
(``sim.cpp``, loaded through ``cxx``), which the GPU tests and the benchmark's
CPU baseline use, and in numpy (``schedules`` and ``orders``).  The two are
independent restatements, cross-checked bit for bit on every collective, and
the pins hold for both.  The pages are:

* the Broadcast/Scatter page, "一对多通信：Broadcast 与 Scatter" (one-to-many
  communication: Broadcast and Scatter), cited below as [Bcast/Scatter page];
* the CSDN article on CANN hccl's AllReduce algorithms, sections "Ring算法",
  "Mesh算法", "Tree算法" and "hccl_allreduce接口详解", cited as [hccl article];
* the latency-formula page, "集合通信算法延迟公式" (alpha-beta latency formulas
  of collective algorithms), cited as [Latency-formula page] with its equation
  labels (e.g. eq. model-algo-ring-ar).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product library never imports, links or calls it,
and it imports nothing from the product library.  It shares no code with the
CUDA path; the only shared module is ``synthetic_inputs`` (seeded numbers, no
collective arithmetic).

Modules:

* ``numerics``   -- fp32 / int32 lane arithmetic and the bf16 <-> fp32 rules.
* ``partition``  -- how a buffer is cut into N chunks.
* ``translog``   -- the transfer log each schedule writes.
* ``cxx``        -- the C++ oracle: every schedule, the closed-form trees and
                    the element conversions (``sim.cpp``, ``sim.h``).
* ``schedules``  -- every algorithm as a message-passing simulation (numpy).
* ``orders``     -- the per-element association tree each algorithm produces,
                    stated in closed form and evaluated for sampled elements.
* ``cost_model`` -- the alpha-beta (Hockney) formulas and busbw factors.

Parity status of each function is stated in its docstring.  Functions whose
exact association order rests on a reading of the pages (not on a printed
table) say so; their data results are still pinned by the definitions.
"""
from . import numerics, partition, translog, schedules, orders, cost_model  # noqa: F401
