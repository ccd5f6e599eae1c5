"""Float64 CPU oracle for GPTQ layer quantization and EoRA compensation.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
library under ``post_weight_quantization_30_b300`` never imports it, and this
package imports nothing from the library: the two share no code.  The only
common dependency is the seeded input generator in ``synthetic``.

Pages followed (cited by title and section throughout):

* [GPTQ-wiki]  "GPTQ" -- wikiprompt.org encyclopedia entry; sections
  "Enfoque Técnico", "Rendimiento y Precisión", "Limitaciones y Alternativas".
* [LowBit]     "El balance de errores de la inferencia de pocos bits: escalas de
  cuantización, calibración y ahorro real de memoria" -- auturnal.com guide;
  sections 1-6 and "Ejemplo resuelto que permite repetir el cálculo".
* [EoRA-blog]  "Aumento de la precisión de LLM de 2 bits con EoRA" -- 7minutos.es;
  sections "Bucear en el espacio propio en busca de un adaptador",
  "Consumo de memoria de Eora".
* [GPTQ-LoRA]  "Resumen Técnico: GPTQ-intrinsic LoRA" -- gist.science 2606.01412;
  "Declaración del Problema" (the layer-wise objective).

The pages never print the GPTQ update equations (the "Ecuaciones fundamentales
y derivaciones" heading of [LowBit] has no body).  The oracle therefore follows
the Optimal-Brain-Quantization lineage that [GPTQ-wiki] "Enfoque Técnico"
names -- greedy compensation by a closed-form update driven by the inverse
Hessian, columns processed in a fixed order -- written out eagerly and
unblocked.  Every reading of an open point is listed in the module docstrings.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against brute force, closed forms or the pages' worked numbers.
"""
from . import eora, gptq, pack, storage  # noqa: F401
