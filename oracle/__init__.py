"""Float64 CPU oracle for paged MLA decode (test infrastructure only; the
product path never imports it)."""
