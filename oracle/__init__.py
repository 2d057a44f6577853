"""fp64 CPU oracle of the routed mixture-of-experts expert computation.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never links, imports or calls it, and it shares no code with the CUDA path:
the two meet only at the seeded inputs from ``synth``.

What it computes (plain definitions, slow, obviously correct):
  * codecs.py  - E2M1 / E8M0 / E4M3 / bf16 / NF3 decoders and encoders and the
                 MXFP8 block quantiser, each written from its bit-field definition;
  * moe.py     - routing by definition (stable counting order), clamped SwiGLU,
                 per-expert weight dequantisation and the MoE forward
                 out[t] = sum_j w[t,j] * expert_{id[t,j]}(x[t]), in two forms
                 (per-expert dgemm, and a brute-force per-token loop).

Parity status of each function is stated in its docstring ("pinned by ...");
every function here is pinned by tests under ``tests/`` that do not re-use it.
"""
