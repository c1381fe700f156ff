"""CPU oracle for the ReplaySSM decode path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 numpy restatement of what the ReplaySSM decode method
computes, written from the pages' description and the published recurrences
of the layer types they name. It exists to check the CUDA path; it is never
part of it. Only the test suite, the package smoke check and the benchmark's
CPU-baseline leg may import, call or execute anything in this package, and
this package imports nothing from the CUDA package.

Sources (cited by page title and section throughout):

* "ReplaySSM: o ganho aparece na carga concorrente, não no nome da
  otimização" -- intro (state = checkpoint + buffer of
  recent inputs), "Cuidados e limites" (outputs equal conventional decoding
  up to floating point; low-precision reads separated from the
  higher-precision recurrence), "O que muda para quem desenvolve" (W = 16,
  FP32 state; speculative acceptance by moving a pointer).
* "NVIDIA y Princeton aceleran modelos híbridos al guardar entradas recientes
  en lugar del estado completo" -- paragraph 2 (append to the
  buffer, output from the checkpoint, consolidate only when the buffer is
  full), paragraph 3 (rollback by a buffer pointer, no per-draft snapshot),
  paragraph 4 (high-precision checkpoint, lower-precision read copy).
* "NVIDIA présente ReplaySSM : accélérer le décodage des modèles hybrides
  Mamba et GDN" -- "Pourquoi les hybrides sont devenus la
  norme" names the three layer types (Mamba-2, Gated DeltaNet, Kimi Delta
  Attention), whose standard decode recurrences are restated here.

Modules:
  recurrences -- conventional per-token recurrences (the primary definition).
  replay      -- the method's replay formulas evaluated naively (self-check).
  method      -- ring / pointer model driving the recurrences call by call.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, an independent published formulation and
brute force (see each test's docstring). No function is "parity unpinned".
"""

from . import method, recurrences, replay  # noqa: F401
