"""fp64 CPU oracle for shared-prompt tree attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of the package entry
point and the CPU-baseline leg of the benchmark may import or run anything in this
package.  The library itself never does: the CUDA path has no CPU fallback.

The oracle shares no code with the CUDA path.  Its inputs come from the seeded
`workloads` module, which holds no attention arithmetic.

Modules:
  attention  - the attention definition (AugTree paper, Sec. 2.2), flattened per
               prompt-response pair (Sec. 2.1; the b=0 ring fallback of Sec. 3.4), a
               tree-direct form over the valid KV context of Eq. 1 (Sec. 3.2) with the
               many-to-one prompt gradient of Eq. 2, a per-row form for sampled rows,
               and the partial-softmax-state merge of Sec. 3.3.
  schedule   - the reference builder of the largest-first tile work queues (replay
               units and greedy balancing, Sec. 3.4).
  invariants - exact identities of attention gradients used for full-size checks.

Every function here is pinned by tests under tests/ (brute force, finite differences,
a library routine with an explicit mask, closed forms and invariants).
"""
