"""CPU oracle for Orca-style iteration-level scheduling with selective batching.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA path; the two meet
only at the seeded inputs drawn by ``iteration_level_scheduling_gb300.synth``.

Everything here is the plain, slow definition of what the method computes,
in float64 NumPy (the pages fix no precision):

* ``kv``        -- per-request maximum-length K/V reservation pool.
* ``sched``     -- iteration-level and request-level schedulers, and the
                   slot-model closed forms they reduce to.
* ``model``     -- one iteration of a pre-LN GPT over a selectively batched
                   mix of initiation and increment requests.
* ``padded``    -- the same iteration computed the padding + masking way.
* ``unbatched`` -- the same iteration run one request at a time.

Citations name the source page and its section.  Page short names:
  [houmin]      garden.houmin.site "Orca" notes (sections 3.1.1-3.1.3)
  [0h-n0]       "論文解説: Orca — Iteration-Level Scheduling..." (0h-n0.github.io)
  [ultralytics] "Continuous Batching" glossary page (ultralytics.com)
  [arcsin2]     "ORCA: A Distributed Serving System for Transformer-Based
                Generative Models" paper notes (arcsin2 / unpurerationalist blog)
  [estelledc]   "Orca — 让一批 LLM 请求随到随走..." study notes (estelledc.github.io)

Parity status: the scheduler, the K/V pool and the flattening are pinned by
the worked examples the pages print; the model iteration is pinned by
library routines (torch CPU layer_norm / gelu / scaled_dot_product_attention /
TransformerEncoderLayer), closed forms and the selective == unbatched ==
padded invariants.  Absolute model outputs on random weights have no printed
value on the pages.
"""
