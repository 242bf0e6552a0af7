"""CPU oracle of the DDP Reducer gradient path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the reducer computes,
written from the pages that describe it:

* "PyTorch Distributed: Experiences on Accelerating Data Parallel Training"
  (arXiv 2006.15704; the paper-graph-ui and paperlayer.ai summaries),
* "Distributed Data Parallel" (tensorplay.cn notes),
* "NCCL 专家课程 30: DDP Reducer、Bucket 与计算通信重叠" (blog.cptz.space),
* "PyTorch Distributed Training Internals" (sandeep007734.github.io).

Modules:
  buckets    -- parameter -> bucket assignment and the locator table
  readiness  -- per-iteration readiness state machine (in-order launch, parking)
  reduce     -- gather into buckets, W-way fp32 mean, copy-back
  nosync     -- local accumulation under no_sync

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the C-ABI library and
its Python binding) never imports, links or calls it, and shares no code
with it.

Parity status: every function here is pinned by ``-m "not gpu"`` tests
against facts the pages or mathematics fix (brute force on tiny inputs,
the pages' layout table and parking sequence, closed forms, exact integer
arithmetic, the Linear(10,10) full-batch identity).  No function is
"parity unpinned".
"""
