"""GB300 speculative verification for block-diffusion LLMs (package stub; bindings follow)."""
