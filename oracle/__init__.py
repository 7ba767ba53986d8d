"""CPU oracle for the batch-invariant MoE layer and the logprob/KL head.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 restatement of
what the hot path computes, written from the source pages' description of the
method.  Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  The CUDA library never calls it and shares no
code, table or helper with it; the two meet only through the seeded input
generators in ``serve_invariant_moe_gb300.synth``, which hold none of the
method's arithmetic.

Sources (cited by page title and section):

* "位级一致：前沿训练的差异化关键" (Fireworks, bit-level agreement for frontier
  training), section "为什么比特级一致是一个复杂的问题" (why bitwise agreement is
  hard): the reductions whose order must be pinned (router, expert matmuls),
  router near-ties and the deterministic tie decision, one kernel choice for the
  expert matmuls whatever the token count.
* "Reinforcement Learning: Why Numerical Alignment and MoE Routing Matter So
  Much" (Fireworks), section "混合专家模型更难对齐" (MoE models are harder to
  align): the k3 divergence, its 0.001 equivalence threshold and the finding
  that the precision and order of the weighted expert combine must match.
* "GLM Post-Training Beyond SFT", section "IcePop 为什么有两层 ratio" (why
  IcePop has two ratios): the mismatch ratio rho_t = pi_train / pi_infer and the
  mask m_t = 1[1/beta <= rho_t <= beta] with beta = 2; sections "迁移到 NPU 时"
  and "动作与概率契约": the top-k tie / order / NaN contract and the
  logsumexp comparison contract.
* Same bit-agreement page, section "端到端零 KLD": the trainer follows the same
  bit-exact standard as the serving path; the head backward here is the chain
  rule of the forward definition, written out.

Modules:
    numerics  -- exact bf16 <-> float64 conversion and round-to-nearest-even.
    moe       -- router logits, top-k with lowest-index ties, gates, SwiGLU
                 experts, dispatch plan invariants, fixed-order combine, and the
                 dense-all-experts-then-mask brute force.
    head      -- vocab projection, log-sum-exp, token logprob, k3, IcePop mask,
                 the IcePop-masked clipped loss and its gradient, DIS weights,
                 and the head backward (dlogits, d hidden, d vocab weights).

Every function here is parity-pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against closed forms, library routines, brute force
on tiny inputs or the pages' own values (``tests/golden/``).
"""
